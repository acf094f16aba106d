// Internal declarations of the GB300 sparse embedding library (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>

#include "emb.h"

namespace emb {

// ---------------------------------------------------------------------------
// sticky device error bits (read and cleared by emb_sync_status)
// ---------------------------------------------------------------------------
enum : int {
    ERRBIT_KEY_RANGE = 1,
    ERRBIT_TABLE_ID = 2,
    ERRBIT_CAPACITY = 4,
    ERRBIT_TIMEOUT = 8,
    ERRBIT_OFFSETS = 16,   // offsets outside [0, nnz] or decreasing: clamped, flagged as a bad argument
};

// Offsets are read clamped into [lo, nnz]: a bad CSR from a caller then never
// sends a kernel outside the keys or the per-lookup workspace.
__device__ __forceinline__ int64_t clamp_offset(int64_t v, int64_t lo, int64_t nnz)
{
    return v < lo ? lo : (v > nnz ? nnz : v);
}

constexpr int kMaxDim = 128;          // dims are multiples of 4 in [4, 128]
constexpr int kMaxTables = 4096;
constexpr uint32_t kEmptySlot = 0xFFFFFFFFu;
constexpr uint32_t kNoSlot = 0xFFFFFFFEu;

// Per-table metadata, resident in device memory.
struct TableDev {
    void* w;             // rows x dim, dtype
    float* state;        // rows x dim fp32 (Adagrad), rows fp32 (row-wise Adagrad) or null
    float* master;       // rows x dim fp32 master copy of a 16-bit table, or null
    int64_t rows;
    uint32_t row_base;   // global row id of row 0
    int32_t dim;
    int32_t dtype;       // emb_dtype
    int32_t pooling;     // emb_pooling
    int32_t opt;         // emb_opt
    float lr, eps;
    int32_t doff;        // column offset in the concatenated output
    int32_t dynamic;     // 1: keys are int64 ids mapped to rows by map_keys
    unsigned long long* map_keys;   // dynamic tables: [rows] key held by each row (kMapEmpty = free)
    const __half* cache_w;          // inference cache: [cache rows][dim] fp16 copies of chosen rows, or null
    const unsigned long long* cache_map;   // open addressing: (row << 32) | cache slot, kCacheEmpty = free
    uint32_t cache_mask;            // cache_map has cache_mask + 1 entries (a power of two)
    int32_t pad2_;
};

// ---------------------------------------------------------------------------
// device helpers shared by the reduction kernels: compensated (Kahan) fp32
// addition, row loads/stores in the table dtype (16-byte fp32 or 8-byte 16-bit
// vectors of 4 columns) and one optimizer step on 4 columns
// ---------------------------------------------------------------------------
__device__ __forceinline__ void kahan_add(float& s, float& c, float x)
{
    float y = __fsub_rn(x, c);
    float t = __fadd_rn(s, y);
    c = __fsub_rn(__fsub_rn(t, s), y);
    s = t;
}

// Packed fp32 pairs: one add.rn.f32x2 / sub.rn.f32x2 / mul.rn.f32x2 rounds
// each half to nearest-even exactly as two scalar __fadd_rn / __fsub_rn /
// __fmul_rn would, in one instruction.
__device__ __forceinline__ float2 add2(float2 a, float2 b)
{
    unsigned long long r;
    asm("add.rn.f32x2 %0, %1, %2;"
        : "=l"(r)
        : "l"(*reinterpret_cast<unsigned long long*>(&a)), "l"(*reinterpret_cast<unsigned long long*>(&b)));
    return *reinterpret_cast<float2*>(&r);
}

__device__ __forceinline__ float2 sub2(float2 a, float2 b)
{
    unsigned long long r;
    asm("sub.rn.f32x2 %0, %1, %2;"
        : "=l"(r)
        : "l"(*reinterpret_cast<unsigned long long*>(&a)), "l"(*reinterpret_cast<unsigned long long*>(&b)));
    return *reinterpret_cast<float2*>(&r);
}

__device__ __forceinline__ float2 mul2(float2 a, float2 b)
{
    unsigned long long r;
    asm("mul.rn.f32x2 %0, %1, %2;"
        : "=l"(r)
        : "l"(*reinterpret_cast<unsigned long long*>(&a)), "l"(*reinterpret_cast<unsigned long long*>(&b)));
    return *reinterpret_cast<float2*>(&r);
}

// kahan_add on two columns at once.
__device__ __forceinline__ void kahan_add2(float2& s, float2& c, float2 x)
{
    const float2 y = sub2(x, c);
    const float2 t = add2(s, y);
    c = sub2(sub2(t, s), y);
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

// What every table of a layer has in common, fixed at compile time where the
// layer is uniform (-1: read from each table's descriptor at run time).
template <int OPT, int DT, int POOL, int MASTER>
struct LayerSpec {
    static constexpr int kOpt = OPT, kDt = DT, kPool = POOL, kMaster = MASTER;
};
using AnyLayer = LayerSpec<-1, -1, -1, -1>;

template <class S>
__device__ __forceinline__ int opt_of(const TableDev& tb) { return S::kOpt >= 0 ? S::kOpt : tb.opt; }
template <class S>
__device__ __forceinline__ int dtype_of(const TableDev& tb) { return S::kDt >= 0 ? S::kDt : tb.dtype; }
template <class S>
__device__ __forceinline__ bool mean_of(const TableDev& tb) { return (S::kPool >= 0 ? S::kPool : tb.pooling) == EMB_POOL_MEAN; }
template <class S>
__device__ __forceinline__ float* master_of(const TableDev& tb) { return S::kMaster == 0 ? nullptr : tb.master; }

// One optimizer step on 4 consecutive elements (starting at elem) of row
// `row`, whose current values have been loaded: w (from load_update_w4), and
// the state a from load_state4.  A table with a master copy gets the new
// fp32 values there and their nearest-even rounding in the stored row.  ssq is the sum over the whole row of G^2 (row-wise Adagrad
// only; the caller reduces it over the lanes holding the row), and `writer`
// says which one lane stores the row's accumulator.
template <class S = AnyLayer>
__device__ __forceinline__ void apply_update4(const TableDev& tb, int64_t row, int64_t elem, const float g[4],
                                              float4 w, float4 a, float ssq, bool writer)
{
    float wv[4] = {w.x, w.y, w.z, w.w};
    const int opt = opt_of<S>(tb);
    if (opt == EMB_OPT_ADAGRAD) {
        float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            av[q] = __fmaf_rn(g[q], g[q], av[q]);
            float den = __fadd_rn(__fsqrt_rn(av[q]), tb.eps);
            wv[q] = __fmaf_rn(-tb.lr, __fdiv_rn(g[q], den), wv[q]);
        }
        *reinterpret_cast<float4*>(tb.state + elem) = make_float4(av[0], av[1], av[2], av[3]);
    } else if (opt == EMB_OPT_ROWWISE_ADAGRAD) {
        const float an = __fadd_rn(a.x, __fdiv_rn(ssq, (float)tb.dim));
        const float den = __fadd_rn(__fsqrt_rn(an), tb.eps);
#pragma unroll
        for (int q = 0; q < 4; ++q) wv[q] = __fmaf_rn(-tb.lr, __fdiv_rn(g[q], den), wv[q]);
        if (writer) tb.state[row] = an;
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) wv[q] = __fmaf_rn(-tb.lr, g[q], wv[q]);
    }
    float* const master = master_of<S>(tb);
    if (master) *reinterpret_cast<float4*>(master + elem) = make_float4(wv[0], wv[1], wv[2], wv[3]);
    store_w4(tb.w, dtype_of<S>(tb), elem, make_float4(wv[0], wv[1], wv[2], wv[3]));
}

// The weights an update starts from: the fp32 master when the table has one,
// else the stored row.
template <class S = AnyLayer>
__device__ __forceinline__ float4 load_update_w4(const TableDev& tb, int64_t elem)
{
    const float* master = master_of<S>(tb);
    if (master) return *reinterpret_cast<const float4*>(master + elem);
    return load_w4(tb.w, dtype_of<S>(tb), elem);
}

// Optimizer state of the 4 elements at elem of row `row`: Adagrad's four
// accumulators, row-wise Adagrad's one (in .x), nothing for SGD.
template <class S = AnyLayer>
__device__ __forceinline__ float4 load_state4(const TableDev& tb, int64_t row, int64_t elem)
{
    const int opt = opt_of<S>(tb);
    if (opt == EMB_OPT_ADAGRAD) return *reinterpret_cast<const float4*>(tb.state + elem);
    if (opt == EMB_OPT_ROWWISE_ADAGRAD) return make_float4(tb.state[row], 0.f, 0.f, 0.f);
    return make_float4(0.f, 0.f, 0.f, 0.f);
}

// Sum of squares of a lane's 4 gradient values.
__device__ __forceinline__ float sq4(const float g[4])
{
    return __fmaf_rn(g[3], g[3], __fmaf_rn(g[2], g[2], __fmaf_rn(g[1], g[1], __fmul_rn(g[0], g[0]))));
}

// Sum of v over aligned groups of `width` lanes (a power of two) by an xor
// butterfly: every lane of a group ends with the same bits.
__device__ __forceinline__ float group_sum(float v, int width, uint32_t mask)
{
    for (int off = 1; off < width; off <<= 1) v = __fadd_rn(v, __shfl_xor_sync(mask, v, off));
    return v;
}

// ---------------------------------------------------------------------------
// radix sort of (key, u32 value) pairs, optionally in independent segments
// ---------------------------------------------------------------------------
constexpr int kSortThreads = 256;
constexpr int kSortItems = 12;
constexpr int kSortTile = kSortThreads * kSortItems;   // 3072-element tiles
constexpr int kSortGroupTiles = 16;                     // tiles per group of the two-level count scan
constexpr int kMaxDigitBits = 10;

struct SortPlan {
    int64_t n_max;       // capacity in elements
    int num_seg_max;     // segments the scratch is sized for
    int bits_max;        // keys < 2^bits_max
    int digit_bits;      // D
    int passes_max;      // ceil(bits_max / D)
    int64_t tiles_max;
    int64_t groups_max;
    size_t scratch_bytes;   // descriptors, per-tile counts and per-group sums of one sort
};

SortPlan make_sort_plan(int64_t n_max, int bits_max, int num_seg_max = 1);

// Bits of the layer sort's table-local keys for tables of at most rows_max
// rows: enough for every row id and for the all-ones key of a skipped lookup
// in a top digit of its own.
int table_sort_bits(int64_t rows_max);

// One sort.  Keys and values move from (keys_in, vals_in) to (keys_out,
// vals_out) through (keys_tmp, vals_tmp), stable, ascending by key.
// n = n_dev ? min(*n_dev, n_host) : n_host; only the low
// (bits_dev ? *bits_dev : plan bits) bits are sorted.  vals_in == nullptr
// means value = index.  key_sub (nullable, plain sorts) is subtracted from
// every key first.
// Segments: with offsets == nullptr the input is one segment.  Otherwise
// segment s ends at clamp(offsets[(s+1)*stride]) (made non-decreasing, the
// last one at n) and each segment is sorted in place.  With `tables` set (the
// layer sort, u32 keys, one segment per table) keys are global row ids: each
// is ranked by its id local to the segment's table, ids at or above
// `sentinel` (or outside the table) rank last and come out as `sentinel`
// behind every valid id of every segment, so the output is the ascending sort
// of the ids.
struct SortArgs {
    const void* keys_in;
    const uint32_t* vals_in;
    void* keys_out;
    uint32_t* vals_out;
    void* keys_tmp;
    uint32_t* vals_tmp;
    int64_t n_host;
    const int64_t* n_dev;
    const int32_t* bits_dev;
    const uint64_t* key_sub;
    const int64_t* offsets;
    int32_t stride;
    int32_t num_seg;
    const TableDev* tables;
    uint32_t sentinel;
    // filled in by radix_sort_pairs from the plan
    int bits_max;
    int D;
    uint64_t skip_key;
};

inline SortArgs sort_args(const void* keys_in, const uint32_t* vals_in, void* keys_out, uint32_t* vals_out,
                          void* keys_tmp, uint32_t* vals_tmp, int64_t n_host)
{
    SortArgs a{};
    a.keys_in = keys_in;
    a.vals_in = vals_in;
    a.keys_out = keys_out;
    a.vals_out = vals_out;
    a.keys_tmp = keys_tmp;
    a.vals_tmp = vals_tmp;
    a.n_host = n_host;
    a.stride = 1;
    a.num_seg = 1;
    return a;
}

// Launches the sort; `scratch` holds plan.scratch_bytes and needs no initial
// contents.  Returns the number of kernels launched, or -1 on a launch error.
template <typename K>
int radix_sort_pairs(const SortPlan& plan, SortArgs a, void* scratch, cudaStream_t st);

// ---------------------------------------------------------------------------
// run-length encoding of sorted keys (unique / counts / segment offsets)
// ---------------------------------------------------------------------------
constexpr int kRleThreads = 256;
constexpr int kRleItems = 16;
constexpr int kRleTile = kRleThreads * kRleItems;

size_t rle_scratch_bytes(int64_t n_max);

// From sorted keys sk[0..n): U runs of keys <= key_max.  Writes
// unique[s] = sk + key_add (int64 or u32 output), seg_off[0..U], counts[0..U),
// inverse[vals[p]] = s (or U for keys > key_max) when inverse != null,
// *num_unique = U, or -1 when *err (nullable) is set by the sort before it.
// Returns kernels launched or -1.
template <typename K>
int rle_sorted(const K* sk, const uint32_t* vals, int64_t n, uint64_t key_max,
               const uint64_t* key_add, int64_t* unique64, uint32_t* unique32,
               int32_t* seg_off, int32_t* counts, int32_t* inverse, int64_t* num_unique,
               void* scratch, const int* err, cudaStream_t st);

// ---------------------------------------------------------------------------
// kernels driven from layer.cu (defined in the other translation units)
// ---------------------------------------------------------------------------
struct ReduceArgs {
    const uint32_t* skeys;      // sorted keys (global ids or unique indices)
    const uint32_t* sbags;      // bag id per sorted position
    int64_t n;
    int64_t chunk;              // nominal positions per warp (starts snap to run starts)
    int64_t nchunks;
    uint32_t key_limit;         // keys >= limit are skipped ...
    const int64_t* key_limit_dev; // ... or >= *key_limit_dev when non-null
    const uint32_t* gid_of_key; // null: key is the global id
    const TableDev* tables;
    int32_t num_tables;
    int32_t batch;
    const float* grad;
    int64_t ld;
    const float* bag_scale;
    float* slots;               // [nchunks][2][kMaxDim]
    uint32_t* split_list;       // [nchunks] chunks where a split run starts (short rows from the front,
                                // rows split over many chunks from the back)
    int* split_count;           // [4] entries of the two lists, then the combine's work counters
    int* long_done;             // [nchunks] segments finished per long split run (zero between backwards)
    int32_t max_dim;            // widest table of the layer (selects the chunk kernel's occupancy)
    int32_t uni_opt, uni_dtype, uni_pool, uni_master;   // shared by every table, or -1 (selects a specialised kernel)
    int* err;
};

int launch_reduce_update(const ReduceArgs& a, cudaStream_t st);   // returns kernels launched or -1

struct FwdArgs {
    const int64_t* keys;
    const int64_t* offsets;
    int64_t nnz;                // keys and per-lookup outputs hold nnz entries; offsets are clamped to it
    const int32_t* table_ids;
    int32_t batch;
    int32_t num_tables;
    float* out;
    int64_t ld;
    const TableDev* tables;
    uint32_t* gid_out;          // global row id per lookup (sentinel when skipped)
    uint32_t* bag_out;          // bag id per lookup
    int64_t* tab_start;         // [T] first lookup of each table (written with the ids)
    float* bag_scale;           // 1/L per mean-pooled bag
    uint32_t sentinel;          // = total rows: sorts after every valid id
    int64_t warps_per_table;
    bool write_ids;             // the pooling kernel also writes gid_out / bag_out
    bool rows16;                // every table stores 16-bit rows (selects the pooling kernel's occupancy)
    const int64_t* resolved;    // dynamic tables: row of each lookup (-1: none), read instead of keys
    bool infer;                 // the inference forward (reads caches, writes nothing for a backward)
    int32_t* order_buf;         // [T] scratch for the tables' processing order, or null
    const int32_t* order;       // set by launch_forward: table of each run of warps (null: table order)
    int* err;
};

int launch_forward(const FwdArgs& a, cudaStream_t st);

// ---------------------------------------------------------------------------
// dynamic tables: int64 keys -> rows through an open-addressing map (dynamic.cu)
// ---------------------------------------------------------------------------
constexpr unsigned long long kMapEmpty = 0x8000000000000000ull;   // the reserved key -2^63

struct DynArgs {
    const int64_t* keys;
    const int64_t* offsets;
    int64_t nnz;
    int32_t batch;
    const TableDev* tables;
    const int32_t* dyn_tables;  // [num_dyn] indices of the dynamic tables
    int32_t num_dyn;
    const float* init_acc;      // [T] initial accumulator values
    uint64_t seed;              // initial values of inserted rows (counter-based, as emb_init_uniform)
    float lo, hi;
    int64_t* resolved;          // [nnz] row of each lookup of a dynamic table (-1: reserved key or map full)
    int* err;
};

// Finds or inserts the key of every lookup of the dynamic tables; a row taken
// for a new key gets its initial values.  Returns kernels launched or -1.
int launch_dyn_resolve(const DynArgs& a, int64_t nnz, cudaStream_t st);
// Rows of n keys of dynamic table t (-1 when absent), without inserting.
int launch_dyn_find(const TableDev* tables, int t, const int64_t* keys, int64_t n, int64_t* rows_out,
                    cudaStream_t st);
// Marks every row of a map free.
int launch_dyn_clear(unsigned long long* map_keys, int64_t rows, cudaStream_t st);

// ---------------------------------------------------------------------------
// inference forward with fp16 caches of chosen rows (infer.cu)
// ---------------------------------------------------------------------------
constexpr unsigned long long kCacheEmpty = ~0ull;

// Fills table t's cache from n row ids (device): slot i holds row rows[i] in
// fp16 (rows held twice keep their first slot); cache_map must be all
// kCacheEmpty.  Returns kernels launched or -1.
int launch_cache_fill(const TableDev& tb, int t, const int64_t* rows, int64_t n, __half* cache_w,
                      unsigned long long* cache_map, uint32_t cache_mask, int* err, cudaStream_t st);

struct InferArgs {
    const int64_t* keys;
    const int64_t* offsets;
    int64_t nnz;
    int32_t batch;
    const TableDev* tables;
    const int32_t* dyn_tables;  // [num_dyn] indices of the dynamic tables
    int32_t num_dyn;
    int64_t* resolved;          // [nnz] row of each lookup of a dynamic table (-1: never seen)
};

// Rows of the dynamic tables' keys for the inference forward, found without
// inserting.  Returns kernels launched or -1.
int launch_infer_resolve(const InferArgs& a, int64_t nnz, cudaStream_t st);
int launch_forward_ids(const FwdArgs& a, cudaStream_t st);   // gid_out / bag_out only

// dedup helpers (dedup.cu); each returns kernels launched or -1
int launch_hash_insert(const uint32_t* gid, int64_t n, uint32_t limit, uint32_t* table, uint32_t mask,
                       uint32_t* slot_of, uint32_t* ukey, uint32_t* uslot, int64_t* ucount, int* err,
                       cudaStream_t st);
int launch_hash_rank_inverse(const uint32_t* sslot, const int64_t* U_dev, uint32_t* slot_rank, int32_t* bits_dev,
                             int32_t* seg_off, const uint32_t* slot_of, int64_t n, uint32_t* inv, cudaStream_t st);
int launch_seg_from_sorted(const uint32_t* sk, int64_t n, const int64_t* U_dev, int32_t* seg_off, int32_t* counts,
                           cudaStream_t st);
int launch_hash_clear(uint32_t* table, const uint32_t* sslot, const int64_t* U_dev, int64_t n_max, cudaStream_t st);
int launch_gather_u32(const uint32_t* src, const uint32_t* idx, int64_t n, uint32_t* dst, cudaStream_t st);
int launch_minmax(const int64_t* keys, int64_t n, unsigned long long* mm, uint64_t* key_sub, int32_t* bits_dev,
                  cudaStream_t st);

}  // namespace emb
