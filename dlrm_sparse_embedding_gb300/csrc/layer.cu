// C ABI of the library: layer life cycle, table initialisation and row I/O,
// and the host drivers of the forward, the three backward variants and the
// stand-alone unique.  Everything the step needs is allocated in emb_create;
// the step itself only launches kernels on the caller's stream.
#include <cstdlib>
#include <cstring>
#include <new>
#include <utility>
#include <vector>

#include "emb_internal.cuh"

using namespace emb;

struct emb_layer {
    int device = 0;
    int32_t T = 0;
    int32_t max_batch = 0;
    int64_t max_nnz = 0;
    std::vector<emb_table_spec> specs;
    std::vector<TableDev> tabs;
    TableDev* d_tables = nullptr;
    uint64_t total_rows = 0;
    int64_t total_dim = 0;
    int32_t maxdim = 0;
    int64_t test_chunk = 0;   // EMB_TEST_REDUCE_CHUNK (0: unset)

    // forward -> backward
    uint32_t* gid = nullptr;
    uint32_t* bag = nullptr;
    float* bag_scale = nullptr;
    // sort buffers
    uint32_t *sk = nullptr, *sv = nullptr, *tk = nullptr, *tv = nullptr;
    void* sort_scratch = nullptr;      // descriptors and counts of one sort (the largest plan's)
    int64_t* tab_start = nullptr;      // [T+1] first lookup of each table in the last forward
    SortPlan plan_gid{}, plan_inv{}, plan_ukey{};
    // dedup results
    int64_t* num_unique = nullptr;
    int32_t* seg_off = nullptr;
    int32_t* cnt = nullptr;
    uint32_t* inverse = nullptr;
    uint32_t* uniq32 = nullptr;
    void* rle_scratch = nullptr;
    // hash dedup
    int64_t max_unique = 0;
    uint32_t* htable = nullptr;
    uint32_t hmask = 0;
    uint32_t* slot_rank = nullptr;
    uint32_t *ukey = nullptr, *uslot = nullptr, *ukey_s = nullptr, *uslot_s = nullptr;
    int32_t* bits_dev = nullptr;
    // segmented reduction
    float* slots = nullptr;
    uint32_t* split_list = nullptr;
    int* split_count = nullptr;
    int* long_done = nullptr;
    int32_t* table_order = nullptr;   // [T] the forward's table processing order
    int64_t nchunks_max = 0;
    int* err = nullptr;
    int64_t* scratch64 = nullptr;   // [2]: num-unique copy target, misc
    // dynamic tables (dynamic.cu)
    int32_t num_dyn = 0;
    int32_t* d_dyn_tables = nullptr;  // [num_dyn]
    float* d_init_acc = nullptr;      // [T]
    int64_t* resolved = nullptr;      // [max_nnz] row of each lookup of a dynamic table
    uint64_t dyn_seed = 0;            // initial values of rows inserted later (last emb_init_uniform)
    float dyn_lo = 0.f, dyn_hi = 0.f;
    // inference caches (infer.cu): per table its fp16 rows and map, freed on rebuild
    std::vector<std::pair<void*, void*>> cache_bufs;

    std::vector<void*> allocs;
    size_t alloc_bytes = 0;

    // step state
    bool fwd_done = false;
    int64_t last_nnz = 0;
    int32_t last_batch = 0;
    bool keep_dedup = false;
    bool dedup_valid = false;
    int32_t dedup_variant = -1;
    const uint32_t* last_unique32 = nullptr;
    const uint32_t* last_sorted_bags = nullptr;
    int64_t launches = 0;

    // dedup run inside emb_forward on an internal stream (-1: off)
    int32_t early_variant = -1;
    cudaStream_t side = nullptr;
    cudaEvent_t ev_in = nullptr, ev_ready = nullptr;
    bool early_pending = false;           // a forward started a dedup on `side`
    int32_t early_pending_variant = -1;
    ReduceArgs early_r{};                 // where that dedup leaves its sorted keys and bags

    // phase timing: events around the forward kernel, the dedup and the
    // reduction, recorded on the streams that run them.  Each step takes the
    // next slot of a ring, and a slot's events are read when the ring comes
    // back to it (or at emb_phase_times), so timing adds no host wait per step.
    bool timing = false;
    struct TimingSlot {
        cudaEvent_t ev[6] = {};           // fwd start/end, dedup start/end, reduce start/end
        bool fwd_pending = false, bwd_pending = false;
    };
    static constexpr int kTimingRing = 64;
    TimingSlot tslot[kTimingRing];
    int tcur = 0;                         // slot of the latest forward
    double phase_ms[EMB_NUM_PHASES] = {0, 0, 0};
    int64_t timed_steps = 0;
};

namespace {

constexpr int64_t kTargetChunks = 65536;
constexpr int64_t kMinChunk = 32, kMaxChunk = 256;

// Nominal lookups per warp in the segmented reduction: enough chunks to fill
// the GPU, at most kMaxChunk so a warp's run list fits in shared memory.
// Nominal lookups per reduction chunk: the smallest power of two in
// [kMinChunk, kMaxChunk] giving at most kTargetChunks chunks.  Tests may
// raise it (EMB_TEST_REDUCE_CHUNK, a power of two in that range, read by
// emb_create) to run the multi-hot chunk kernels on small inputs.
int64_t chunk_for(int64_t n, int64_t at_least = 0)
{
    int64_t c = kMinChunk;
    while (c < kMaxChunk && (c * kTargetChunks < n || c < at_least)) c <<= 1;
    return c;
}

int64_t test_reduce_chunk()
{
    const char* v = std::getenv("EMB_TEST_REDUCE_CHUNK");
    if (!v) return 0;
    const long long c = std::strtoll(v, nullptr, 10);
    return (c >= kMinChunk && c <= kMaxChunk && (c & (c - 1)) == 0) ? (int64_t)c : 0;
}

int64_t nchunks_bound(int64_t max_nnz)
{
    const int64_t big = (max_nnz + kMaxChunk - 1) / kMaxChunk;
    return (big > kTargetChunks ? big : kTargetChunks) + 1;
}

int bits_for(uint64_t max_value)   // bits to hold values 0..max_value
{
    int b = 1;
    while (b < 64 && (max_value >> b) != 0) ++b;
    return b;
}

// Optional cap on what one emb_create may allocate, to exercise the
// out-of-memory path in tests (EMB_TEST_ALLOC_LIMIT_BYTES; unset = no cap).
bool dalloc(emb_layer* L, void** p, size_t bytes)
{
    if (bytes == 0) bytes = 16;
    const char* cap = std::getenv("EMB_TEST_ALLOC_LIMIT_BYTES");
    if (cap && L->alloc_bytes + bytes > (size_t)std::strtoull(cap, nullptr, 10)) return false;
    if (cudaMalloc(p, bytes) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    L->alloc_bytes += bytes;
    L->allocs.push_back(*p);
    return true;
}

template <typename T>
bool dalloc_n(emb_layer* L, T** p, int64_t n)
{
    return dalloc(L, reinterpret_cast<void**>(p), sizeof(T) * (size_t)(n > 0 ? n : 1));
}

void free_all(emb_layer* L)
{
    for (void* p : L->allocs) cudaFree(p);
    L->allocs.clear();
}

size_t dtype_bytes(int32_t dt) { return dt == EMB_F32 ? 4 : 2; }

// fp32 optimizer state values per row: dim (Adagrad), 1 (row-wise Adagrad), 0 (SGD)
int64_t state_cols(const TableDev& d)
{
    return d.opt == EMB_OPT_ADAGRAD ? d.dim : (d.opt == EMB_OPT_ROWWISE_ADAGRAD ? 1 : 0);
}

cudaStream_t S(void* s) { return static_cast<cudaStream_t>(s); }

int track(emb_layer* L, int launched)
{
    if (launched < 0) return EMB_ERR_CUDA;
    L->launches += launched;
    return EMB_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// p is a multiple of a bytes (a power of two); a null pointer passes, its
// presence is checked separately.  A device array misaligned for its element
// type would fault the kernel that reads it, so the host rejects it first.
bool aligned_to(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// ------------------------------- kernels ----------------------------------

__global__ void init_uniform_kernel(void* w, int dtype, int64_t rows, int dim, int t, uint64_t seed, float lo,
                                    float hi, float* state, int state_cols, float init_acc, float* master)
{
    const int64_t total = rows * dim;
    const float d = __fsub_rn(hi, lo);
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = e / dim;
        const int c = (int)(e - r * dim);
        // splitmix64 output number n of the stream started from `seed`
        const uint64_t n = ((uint64_t)t << 44) | ((uint64_t)r << 12) | (uint64_t)c;
        uint64_t z = seed + (n + 1ull) * 0x9E3779B97F4A7C15ull;
        z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
        z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
        z ^= z >> 31;
        const float f = __fmul_rn(__uint2float_rn((uint32_t)(z >> 40)), 5.9604644775390625e-08f);
        const float v = __fadd_rn(lo, __fmul_rn(d, f));
        if (master) master[e] = v;
        if (dtype == EMB_F32) static_cast<float*>(w)[e] = v;
        else if (dtype == EMB_F16) static_cast<__half*>(w)[e] = __float2half_rn(v);
        else static_cast<__nv_bfloat16*>(w)[e] = __float2bfloat16_rn(v);
        if (state && c < state_cols) state[r * state_cols + c] = init_acc;
    }
}

__global__ void gather_rows_kernel(const void* w, const float* state, int state_cols, int dtype, int64_t rows,
                                   int dim, const int64_t* ids, int64_t n, void* wout, float* sout, int* err)
{
    const int64_t total = n * dim;
    const size_t eb = dtype == EMB_F32 ? 4 : 2;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = e / dim;
        const int c = (int)(e - i * dim);
        const int64_t r = ids[i];
        if (r < 0 || r >= rows) {
            if (c == 0) atomicOr(err, ERRBIT_KEY_RANGE);
            continue;
        }
        const int64_t src = r * dim + c;
        if (eb == 4) static_cast<float*>(wout)[e] = static_cast<const float*>(w)[src];
        else static_cast<unsigned short*>(wout)[e] = static_cast<const unsigned short*>(w)[src];
        if (sout && state && c < state_cols) sout[i * state_cols + c] = state[r * state_cols + c];
    }
}

__global__ void widen_u32(const uint32_t* __restrict__ src, const int64_t* __restrict__ n_dev, int64_t n_max,
                          int64_t* __restrict__ dst)
{
    const int64_t n = *n_dev;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n && i < n_max;
         i += (int64_t)gridDim.x * blockDim.x)
        dst[i] = src[i];
}

unsigned grid_for(int64_t n, int threads, int64_t cap = 16384)
{
    int64_t b = (n + threads - 1) / threads;
    if (b < 1) b = 1;
    if (b > cap) b = cap;
    return (unsigned)b;
}

// workspace layout of emb_unique
struct UniqueWs {
    uint64_t *k_tmp, *k_out;
    uint32_t *v_tmp, *v_out;
    void* sort_scratch;
    int32_t* seg;
    void* rle;
    unsigned long long* mm;
    uint64_t* key_sub;
    int32_t* bits;
    size_t total;
};

UniqueWs unique_ws_layout(int64_t n, char* base)
{
    UniqueWs w{};
    size_t off = 0;
    auto take = [&](size_t bytes) -> char* {
        char* p = base ? base + off : nullptr;
        off += (bytes + 255) & ~size_t(255);
        return p;
    };
    const int64_t m = n > 0 ? n : 1;
    SortPlan plan = make_sort_plan(m, 64);
    w.k_tmp = reinterpret_cast<uint64_t*>(take(sizeof(uint64_t) * m));
    w.k_out = reinterpret_cast<uint64_t*>(take(sizeof(uint64_t) * m));
    w.v_tmp = reinterpret_cast<uint32_t*>(take(sizeof(uint32_t) * m));
    w.v_out = reinterpret_cast<uint32_t*>(take(sizeof(uint32_t) * m));
    w.sort_scratch = take(plan.scratch_bytes);
    w.seg = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * (m + 1)));
    w.rle = take(rle_scratch_bytes(m));
    w.mm = reinterpret_cast<unsigned long long*>(take(2 * sizeof(unsigned long long)));
    w.key_sub = reinterpret_cast<uint64_t*>(take(sizeof(uint64_t)));
    w.bits = reinterpret_cast<int32_t*>(take(sizeof(int32_t)));
    w.total = off;
    return w;
}

// Folds the events of one ring slot into the totals (waits for them).
void harvest_slot(emb_layer* L, emb_layer::TimingSlot& s)
{
    float ms = 0.f;
    if (s.fwd_pending) {
        if (cudaEventSynchronize(s.ev[1]) == cudaSuccess && cudaEventElapsedTime(&ms, s.ev[0], s.ev[1]) == cudaSuccess)
            L->phase_ms[EMB_PHASE_FORWARD] += ms;
        s.fwd_pending = false;
    }
    if (s.bwd_pending) {
        if (cudaEventSynchronize(s.ev[5]) == cudaSuccess) {
            if (cudaEventElapsedTime(&ms, s.ev[2], s.ev[3]) == cudaSuccess) L->phase_ms[EMB_PHASE_DEDUP] += ms;
            if (cudaEventElapsedTime(&ms, s.ev[4], s.ev[5]) == cudaSuccess)
                L->phase_ms[EMB_PHASE_REDUCE_UPDATE] += ms;
        }
        s.bwd_pending = false;
        L->timed_steps += 1;
    }
    cudaGetLastError();
}

// Folds every slot still holding events, oldest first.
void harvest_timing(emb_layer* L)
{
    for (int i = 1; i <= emb_layer::kTimingRing; ++i) harvest_slot(L, L->tslot[(L->tcur + i) % emb_layer::kTimingRing]);
}

// The slot a forward records into: the next one of the ring, its old events read first.
emb_layer::TimingSlot& next_timing_slot(emb_layer* L)
{
    L->tcur = (L->tcur + 1) % emb_layer::kTimingRing;
    emb_layer::TimingSlot& s = L->tslot[L->tcur];
    harvest_slot(L, s);
    return s;
}

}  // namespace

namespace emb {

// Host checks of emb_unique's arguments (shared with emb_unique_noalloc):
// sizes, presence and the alignment of every array to its element type.
bool unique_args_valid(const int64_t* keys, int64_t n, const int64_t* unique, const int32_t* inverse,
                       const int32_t* counts, const int32_t* seg_offsets, const int64_t* num_unique)
{
    if (n < 0 || n >= (int64_t(1) << 31) || !num_unique || (n > 0 && (!keys || !unique || !inverse || !counts)))
        return false;
    return aligned_to(keys, 8) && aligned_to(unique, 8) && aligned_to(num_unique, 8) && aligned_to(inverse, 4) &&
           aligned_to(counts, 4) && aligned_to(seg_offsets, 4);
}

}  // namespace emb

extern "C" {

const char* emb_status_string(int status)
{
    switch (status) {
        case EMB_OK: return "ok";
        case EMB_ERR_INVALID_ARG: return "invalid argument";
        case EMB_ERR_OOM: return "out of device memory";
        case EMB_ERR_CUDA: return "CUDA error";
        case EMB_ERR_KEY_RANGE: return "key outside [0, rows)";
        case EMB_ERR_CAPACITY: return "hash table full";
        case EMB_ERR_TIMEOUT: return "bounded wait gave up";
        case EMB_ERR_STATE: return "call out of order";
        default: return "unknown status";
    }
}

int emb_create(const emb_table_spec* specs, int32_t num_tables, int32_t max_batch, int64_t max_nnz,
               emb_layer** out)
{
    if (!specs || !out || num_tables < 1 || num_tables > kMaxTables || max_batch < 1 || max_nnz < 0 ||
        max_nnz >= (int64_t(1) << 31) || (int64_t)num_tables * max_batch >= (int64_t(1) << 31))
        return EMB_ERR_INVALID_ARG;
    uint64_t total_rows = 0;
    int64_t total_dim = 0;
    int32_t maxdim = 0;
    for (int t = 0; t < num_tables; ++t) {
        const emb_table_spec& s = specs[t];
        if (s.rows < 1 || s.dim < 4 || s.dim > kMaxDim || (s.dim & 3) || s.dtype < 0 || s.dtype > 2 ||
            s.pooling < 0 || s.pooling > 1 || s.opt < 0 || s.opt > 2 || s.master_fp32 < 0 || s.master_fp32 > 1 ||
            (s.master_fp32 && s.dtype == EMB_F32) || s.dynamic < 0 || s.dynamic > 1)
            return EMB_ERR_INVALID_ARG;
        total_rows += (uint64_t)s.rows;
        total_dim += s.dim;
        if (s.dim > maxdim) maxdim = s.dim;
    }
    if (total_rows >= 0xFFFFFFFFull) return EMB_ERR_INVALID_ARG;

    emb_layer* L = new (std::nothrow) emb_layer();
    if (!L) return EMB_ERR_OOM;
    cudaGetDevice(&L->device);
    L->T = num_tables;
    L->max_batch = max_batch;
    L->max_nnz = max_nnz;
    L->specs.assign(specs, specs + num_tables);
    L->total_rows = total_rows;
    L->total_dim = total_dim;
    L->maxdim = maxdim;
    L->test_chunk = test_reduce_chunk();

    bool ok = true;
    uint64_t rb = 0;
    int32_t doff = 0;
    L->tabs.resize(num_tables);
    L->cache_bufs.assign(num_tables, std::make_pair(nullptr, nullptr));
    for (int t = 0; t < num_tables && ok; ++t) {
        const emb_table_spec& s = specs[t];
        TableDev& d = L->tabs[t];
        d.rows = s.rows;
        d.row_base = (uint32_t)rb;
        d.dim = s.dim;
        d.dtype = s.dtype;
        d.pooling = s.pooling;
        d.opt = s.opt;
        d.lr = s.lr;
        d.eps = s.eps;
        d.doff = doff;
        d.dynamic = s.dynamic;
        d.map_keys = nullptr;
        d.cache_w = nullptr;
        d.cache_map = nullptr;
        d.cache_mask = 0;
        d.pad2_ = 0;
        d.w = nullptr;
        d.state = nullptr;
        d.master = nullptr;
        ok = dalloc(L, &d.w, (size_t)s.rows * s.dim * dtype_bytes(s.dtype));
        if (ok && state_cols(d) > 0) ok = dalloc_n(L, &d.state, s.rows * state_cols(d));
        if (ok && s.master_fp32) ok = dalloc_n(L, &d.master, s.rows * (int64_t)s.dim);
        if (ok && s.dynamic) ok = dalloc_n(L, &d.map_keys, s.rows);
        rb += (uint64_t)s.rows;
        doff += s.dim;
    }
    const int64_t n = max_nnz;
    L->max_unique = n < (int64_t)total_rows ? n : (int64_t)total_rows;
    const int gid_bits = bits_for(total_rows);                 // ids 0..total_rows (sentinel)
    int64_t rows_max = 1;
    for (int t = 0; t < num_tables; ++t) rows_max = specs[t].rows > rows_max ? specs[t].rows : rows_max;
    // the lookups' ids are sorted table by table on their table-local row
    L->plan_gid = make_sort_plan(n, table_sort_bits(rows_max), num_tables);
    L->plan_ukey = make_sort_plan(L->max_unique, gid_bits);
    L->plan_inv = make_sort_plan(n, bits_for((uint64_t)L->max_unique));
    size_t sort_scratch_bytes = L->plan_gid.scratch_bytes;
    for (const SortPlan* pl : {&L->plan_inv, &L->plan_ukey})
        if (pl->scratch_bytes > sort_scratch_bytes) sort_scratch_bytes = pl->scratch_bytes;
    uint64_t cap = 1024;
    while (cap < 2 * (uint64_t)(L->max_unique > 0 ? L->max_unique : 1)) cap <<= 1;
    L->hmask = (uint32_t)(cap - 1);
    L->nchunks_max = nchunks_bound(n);

    ok = ok && dalloc_n(L, &L->d_tables, num_tables) && dalloc_n(L, &L->gid, n) && dalloc_n(L, &L->bag, n) &&
         dalloc_n(L, &L->bag_scale, (int64_t)num_tables * max_batch) && dalloc_n(L, &L->sk, n) &&
         dalloc_n(L, &L->sv, n) && dalloc_n(L, &L->tk, n) && dalloc_n(L, &L->tv, n) &&
         dalloc(L, &L->sort_scratch, sort_scratch_bytes) && dalloc_n(L, &L->tab_start, num_tables + 1) &&
         dalloc_n(L, &L->num_unique, 1) &&
         dalloc_n(L, &L->seg_off, n + 1) && dalloc_n(L, &L->cnt, n) && dalloc_n(L, &L->inverse, n) &&
         dalloc_n(L, &L->uniq32, n) && dalloc(L, &L->rle_scratch, rle_scratch_bytes(n)) &&
         dalloc_n(L, &L->htable, (int64_t)cap) && dalloc_n(L, &L->slot_rank, (int64_t)cap) &&
         dalloc_n(L, &L->ukey, L->max_unique) && dalloc_n(L, &L->uslot, L->max_unique) &&
         dalloc_n(L, &L->ukey_s, L->max_unique) && dalloc_n(L, &L->uslot_s, L->max_unique) &&
         dalloc_n(L, &L->bits_dev, 1) && dalloc_n(L, &L->slots, L->nchunks_max * 2 * kMaxDim) &&
         dalloc_n(L, &L->split_list, L->nchunks_max) && dalloc_n(L, &L->split_count, 4) &&
         dalloc_n(L, &L->long_done, L->nchunks_max) && dalloc_n(L, &L->table_order, num_tables) &&
         dalloc_n(L, &L->err, 1) && dalloc_n(L, &L->scratch64, 2) && dalloc_n(L, &L->d_init_acc, num_tables);
    std::vector<int32_t> dyn;
    std::vector<float> init_acc(num_tables);
    for (int t = 0; t < num_tables; ++t) {
        if (specs[t].dynamic) dyn.push_back(t);
        init_acc[t] = specs[t].init_acc;
    }
    L->num_dyn = (int32_t)dyn.size();
    if (ok && L->num_dyn > 0)
        ok = dalloc_n(L, &L->d_dyn_tables, L->num_dyn) && dalloc_n(L, &L->resolved, n);
    if (ok) {
        ok = cudaMemcpy(L->d_tables, L->tabs.data(), sizeof(TableDev) * num_tables, cudaMemcpyHostToDevice) ==
                 cudaSuccess &&
             cudaMemset(L->htable, 0xFF, sizeof(uint32_t) * cap) == cudaSuccess &&
             cudaMemset(L->err, 0, sizeof(int)) == cudaSuccess &&
             cudaMemset(L->long_done, 0, sizeof(int) * L->nchunks_max) == cudaSuccess &&
             cudaMemcpy(L->d_init_acc, init_acc.data(), sizeof(float) * num_tables, cudaMemcpyHostToDevice) ==
                 cudaSuccess &&
             (L->num_dyn == 0 || cudaMemcpy(L->d_dyn_tables, dyn.data(), sizeof(int32_t) * L->num_dyn,
                                            cudaMemcpyHostToDevice) == cudaSuccess);
        for (int t = 0; t < num_tables && ok; ++t)
            if (L->tabs[t].dynamic) ok = launch_dyn_clear(L->tabs[t].map_keys, L->tabs[t].rows, 0) >= 0;
        ok = ok && cudaDeviceSynchronize() == cudaSuccess;
        if (!ok) {
            cudaGetLastError();
            free_all(L);
            delete L;
            return EMB_ERR_CUDA;
        }
    }
    if (!ok) {
        free_all(L);
        delete L;
        return EMB_ERR_OOM;
    }
    *out = L;
    return EMB_OK;
}

int emb_destroy(emb_layer* L)
{
    if (!L) return EMB_OK;
    cudaDeviceSynchronize();
    for (auto& s : L->tslot)
        for (cudaEvent_t& e : s.ev)
            if (e) cudaEventDestroy(e);
    if (L->ev_in) cudaEventDestroy(L->ev_in);
    if (L->ev_ready) cudaEventDestroy(L->ev_ready);
    if (L->side) cudaStreamDestroy(L->side);
    for (auto& cb : L->cache_bufs) {
        if (cb.first) cudaFree(cb.first);
        if (cb.second) cudaFree(cb.second);
    }
    free_all(L);
    delete L;
    return EMB_OK;
}

int emb_init_uniform(emb_layer* L, uint64_t seed, float lo, float hi, void* stream)
{
    if (!L) return EMB_ERR_INVALID_ARG;
    L->dyn_seed = seed;
    L->dyn_lo = lo;
    L->dyn_hi = hi;
    for (int t = 0; t < L->T; ++t) {
        const TableDev& d = L->tabs[t];
        if (d.dynamic) {   // rows get their values when a key first takes them
            if (launch_dyn_clear(d.map_keys, d.rows, S(stream)) < 0) return EMB_ERR_CUDA;
            L->launches += 1;
            continue;
        }
        const int64_t total = d.rows * d.dim;
        init_uniform_kernel<<<grid_for(total, 256, 65536), 256, 0, S(stream)>>>(
            d.w, d.dtype, d.rows, d.dim, t, seed, lo, hi, d.state, (int)state_cols(d), L->specs[t].init_acc,
            d.master);
        L->launches += 1;
    }
    return cudaGetLastError() == cudaSuccess ? EMB_OK : EMB_ERR_CUDA;
}

// Launches the dedup of `variant` over the ids in L->gid / L->bag on st and
// points r at its sorted keys and bags (plus the unique-index mapping for the
// hash variant).  Records the by-product pointers for emb_dedup_result.
static int launch_dedup(emb_layer* L, int32_t variant, int64_t n, cudaStream_t st, ReduceArgs& r)
{
    const uint32_t limit = (uint32_t)L->total_rows;
    int rc = EMB_OK;
    r.key_limit = limit;
    r.key_limit_dev = nullptr;
    r.gid_of_key = nullptr;
    // the lookups' ids, table by table (the forward wrote each table's first lookup)
    SortArgs by_table = sort_args(L->gid, L->bag, L->sk, L->sv, L->tk, L->tv, n);
    by_table.offsets = L->tab_start;
    by_table.num_seg = L->T;
    by_table.tables = L->d_tables;
    by_table.sentinel = limit;
    if (variant == EMB_BWD_REDUCTION) {
        rc = track(L, radix_sort_pairs<uint32_t>(L->plan_gid, by_table, L->sort_scratch, st));
        if (rc == EMB_OK && L->keep_dedup)
            rc = track(L, rle_sorted<uint32_t>(L->sk, nullptr, n, limit - 1u, nullptr, nullptr, L->uniq32, L->seg_off,
                                               L->cnt, nullptr, L->num_unique, L->rle_scratch, nullptr, st));
        r.skeys = L->sk;
        r.sbags = L->sv;
        L->last_unique32 = L->uniq32;
        L->last_sorted_bags = L->sv;
    } else if (variant == EMB_BWD_UNIQUE_SORT) {
        by_table.vals_in = nullptr;   // values: positions, for the inverse
        rc = track(L, radix_sort_pairs<uint32_t>(L->plan_gid, by_table, L->sort_scratch, st));
        if (rc == EMB_OK)
            rc = track(L, rle_sorted<uint32_t>(L->sk, L->sv, n, limit - 1u, nullptr, nullptr, L->uniq32, L->seg_off,
                                               L->cnt, reinterpret_cast<int32_t*>(L->inverse), L->num_unique,
                                               L->rle_scratch, nullptr, st));
        if (rc == EMB_OK) rc = track(L, launch_gather_u32(L->bag, L->sv, n, L->tv, st));
        r.skeys = L->sk;
        r.sbags = L->tv;
        L->last_unique32 = L->uniq32;
        L->last_sorted_bags = L->tv;
    } else {
        uint32_t* slot_of = L->sk;   // dead before the second sort writes sk
        rc = track(L, launch_hash_insert(L->gid, n, limit, L->htable, L->hmask, slot_of, L->ukey, L->uslot,
                                         L->num_unique, L->err, st));
        const int64_t umax = n < L->max_unique ? n : L->max_unique;
        if (rc == EMB_OK) {
            SortArgs sa = sort_args(L->ukey, L->uslot, L->ukey_s, L->uslot_s, L->tk, L->tv, umax);
            sa.n_dev = L->num_unique;
            rc = track(L, radix_sort_pairs<uint32_t>(L->plan_ukey, sa, L->sort_scratch, st));
        }
        if (rc == EMB_OK)
            rc = track(L, launch_hash_rank_inverse(L->uslot_s, L->num_unique, L->slot_rank, L->bits_dev, L->seg_off,
                                                   slot_of, n, L->inverse, st));
        if (rc == EMB_OK) {
            SortArgs sa = sort_args(L->inverse, L->bag, L->sk, L->sv, L->tk, L->tv, n);
            sa.bits_dev = L->bits_dev;
            rc = track(L, radix_sort_pairs<uint32_t>(L->plan_inv, sa, L->sort_scratch, st));
        }
        if (rc == EMB_OK) rc = track(L, launch_seg_from_sorted(L->sk, n, L->num_unique, L->seg_off, L->cnt, st));
        r.skeys = L->sk;
        r.sbags = L->sv;
        r.key_limit_dev = L->num_unique;
        r.gid_of_key = L->ukey_s;
        L->last_unique32 = L->ukey_s;
        L->last_sorted_bags = L->sv;
    }
    return rc;
}

int emb_forward(emb_layer* L, const int64_t* keys, const int64_t* offsets, const int32_t* table_ids, int64_t nnz,
                int32_t batch, float* out, void* stream)
{
    if (!L || !offsets || !table_ids || !out || batch < 1 || batch > L->max_batch || nnz < 0 || nnz > L->max_nnz ||
        (nnz > 0 && !keys) || !aligned16(out) || !aligned_to(keys, 8) || !aligned_to(offsets, 8) ||
        !aligned_to(table_ids, 4))
        return EMB_ERR_INVALID_ARG;
    cudaStream_t st = S(stream);
    FwdArgs a;
    a.keys = keys;
    a.offsets = offsets;
    a.nnz = nnz;
    a.table_ids = table_ids;
    a.batch = batch;
    a.num_tables = L->T;
    a.out = out;
    a.ld = L->total_dim;
    a.tables = L->d_tables;
    a.gid_out = L->gid;
    a.bag_out = L->bag;
    a.tab_start = L->tab_start;
    a.bag_scale = L->bag_scale;
    a.sentinel = (uint32_t)L->total_rows;
    a.warps_per_table = (batch + 31) / 32;
    a.order_buf = L->table_order;
    a.write_ids = true;
    a.rows16 = true;
    a.resolved = L->resolved;
    a.infer = false;
    for (const TableDev& d : L->tabs) a.rows16 = a.rows16 && d.dtype != EMB_F32;
    a.err = L->err;
    cudaEvent_t* ev = L->timing ? next_timing_slot(L).ev : nullptr;
    int rc = EMB_OK;
    // a dedup a previous forward left running on the side stream still reads
    // the ids and resolved rows this forward rewrites
    if (L->early_pending && cudaStreamWaitEvent(st, L->ev_ready, 0) != cudaSuccess) return EMB_ERR_CUDA;
    if (ev) cudaEventRecord(ev[0], st);   // the forward phase includes resolving dynamic keys
    if (L->num_dyn > 0 && nnz > 0) {
        // dynamic tables: find or insert every key; the kernels after it read rows
        DynArgs da;
        da.keys = keys;
        da.offsets = offsets;
        da.nnz = nnz;
        da.batch = batch;
        da.tables = L->d_tables;
        da.dyn_tables = L->d_dyn_tables;
        da.num_dyn = L->num_dyn;
        da.init_acc = L->d_init_acc;
        da.seed = L->dyn_seed;
        da.lo = L->dyn_lo;
        da.hi = L->dyn_hi;
        da.resolved = L->resolved;
        da.err = L->err;
        rc = track(L, launch_dyn_resolve(da, nnz, st));
        if (rc != EMB_OK) return rc;
    }
    const bool early = L->early_variant >= 0 && nnz > 0;
    if (early) {
        // ids + dedup on the side stream, concurrent with the pooling kernel
        a.write_ids = false;
        if (cudaEventRecord(L->ev_in, st) != cudaSuccess || cudaStreamWaitEvent(L->side, L->ev_in, 0) != cudaSuccess)
            return EMB_ERR_CUDA;
        if (ev) cudaEventRecord(ev[2], L->side);
        rc = track(L, launch_forward_ids(a, L->side));
        L->early_r = ReduceArgs{};
        if (rc == EMB_OK) rc = launch_dedup(L, L->early_variant, nnz, L->side, L->early_r);
        if (ev) cudaEventRecord(ev[3], L->side);
        if (rc == EMB_OK && cudaEventRecord(L->ev_ready, L->side) != cudaSuccess) rc = EMB_ERR_CUDA;
        if (rc != EMB_OK) return rc;
    }
    rc = track(L, launch_forward(a, st));
    if (ev && rc == EMB_OK) {
        cudaEventRecord(ev[1], st);
        L->tslot[L->tcur].fwd_pending = true;
    }
    if (rc != EMB_OK) return rc;
    L->fwd_done = true;
    L->last_nnz = nnz;
    L->last_batch = batch;
    L->dedup_valid = false;
    L->early_pending = early;
    L->early_pending_variant = early ? L->early_variant : -1;
    return EMB_OK;
}

int emb_set_keep_dedup(emb_layer* L, int32_t keep)
{
    if (!L) return EMB_ERR_INVALID_ARG;
    L->keep_dedup = keep != 0;
    return EMB_OK;
}

int emb_set_early_dedup(emb_layer* L, int32_t variant)
{
    if (!L || variant < -1 || variant > 2) return EMB_ERR_INVALID_ARG;
    if (variant >= 0 && !L->side) {
        if (cudaStreamCreateWithFlags(&L->side, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&L->ev_in, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&L->ev_ready, cudaEventDisableTiming) != cudaSuccess) {
            cudaGetLastError();
            return EMB_ERR_CUDA;
        }
    }
    L->early_variant = variant;
    return EMB_OK;
}

int emb_backward_update(emb_layer* L, const float* grad_out, int32_t variant, void* stream)
{
    if (!L || !grad_out || !aligned16(grad_out) || variant < 0 || variant > 2) return EMB_ERR_INVALID_ARG;
    if (!L->fwd_done) return EMB_ERR_STATE;
    cudaStream_t st = S(stream);
    const int64_t n = L->last_nnz;
    ReduceArgs r{};
    r.n = n;
    r.chunk = chunk_for(n, L->test_chunk);
    r.nchunks = (n + r.chunk - 1) / r.chunk;
    r.tables = L->d_tables;
    r.num_tables = L->T;
    r.batch = L->last_batch;
    r.grad = grad_out;
    r.ld = L->total_dim;
    r.bag_scale = L->bag_scale;
    r.slots = L->slots;
    r.split_list = L->split_list;
    r.split_count = L->split_count;
    r.long_done = L->long_done;
    r.max_dim = L->maxdim;
    r.uni_opt = L->tabs[0].opt;
    r.uni_dtype = L->tabs[0].dtype;
    r.uni_pool = L->tabs[0].pooling;
    r.uni_master = L->tabs[0].master ? 1 : 0;
    for (const TableDev& d : L->tabs) {
        if (d.opt != r.uni_opt) r.uni_opt = -1;
        if (d.dtype != r.uni_dtype) r.uni_dtype = -1;
        if (d.pooling != r.uni_pool) r.uni_pool = -1;
        if ((d.master ? 1 : 0) != r.uni_master) r.uni_master = -1;
    }
    r.err = L->err;
    int rc = EMB_OK;
    L->dedup_valid = false;
    emb_layer::TimingSlot* ts = nullptr;
    if (L->timing) {
        ts = &L->tslot[L->tcur];
        if (ts->bwd_pending) harvest_slot(L, *ts);   // a second backward after one forward
    }
    cudaEvent_t* ev = ts ? ts->ev : nullptr;
    if (n == 0) {
        if (cudaMemsetAsync(L->num_unique, 0, sizeof(int64_t), st) != cudaSuccess ||
            cudaMemsetAsync(L->seg_off, 0, sizeof(int32_t), st) != cudaSuccess)
            return EMB_ERR_CUDA;
        L->dedup_valid = true;
        L->dedup_variant = variant;
        L->last_unique32 = L->uniq32;
        L->last_sorted_bags = L->sv;
        return EMB_OK;
    }
    if (L->early_pending) {
        // the ids (and maybe the dedup) were produced on the side stream
        if (cudaStreamWaitEvent(st, L->ev_ready, 0) != cudaSuccess) return EMB_ERR_CUDA;
    }
    if (L->early_pending && L->early_pending_variant == variant) {
        r.skeys = L->early_r.skeys;
        r.sbags = L->early_r.sbags;
        r.key_limit = L->early_r.key_limit;
        r.key_limit_dev = L->early_r.key_limit_dev;
        r.gid_of_key = L->early_r.gid_of_key;
    } else {
        if (ev) cudaEventRecord(ev[2], st);
        rc = launch_dedup(L, variant, n, st, r);
        if (ev) cudaEventRecord(ev[3], st);
    }
    L->early_pending = false;
    if (ev) cudaEventRecord(ev[4], st);
    if (rc == EMB_OK) rc = track(L, launch_reduce_update(r, st));
    if (rc == EMB_OK && variant == EMB_BWD_UNIQUE_HASH)
        rc = track(L, launch_hash_clear(L->htable, L->uslot_s, L->num_unique, n, st));
    if (ev && rc == EMB_OK) {
        cudaEventRecord(ev[5], st);
        ts->bwd_pending = true;
    }
    if (rc != EMB_OK) return rc;
    L->dedup_valid = variant != EMB_BWD_REDUCTION || L->keep_dedup;
    L->dedup_variant = variant;
    return EMB_OK;
}

int emb_dedup_result(emb_layer* L, int64_t* unique, int32_t* inverse, int32_t* counts, int32_t* seg_offsets,
                     int32_t* sorted_bags, int64_t* num_unique_host, void* stream)
{
    if (!L || !aligned_to(unique, 8) || !aligned_to(inverse, 4) || !aligned_to(counts, 4) ||
        !aligned_to(seg_offsets, 4) || !aligned_to(sorted_bags, 4))
        return EMB_ERR_INVALID_ARG;
    if (!L->dedup_valid) return EMB_ERR_STATE;
    if (inverse && L->dedup_variant == EMB_BWD_REDUCTION) return EMB_ERR_STATE;
    cudaStream_t st = S(stream);
    int64_t U = 0;
    if (cudaMemcpyAsync(&U, L->num_unique, sizeof(int64_t), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return EMB_ERR_CUDA;
    const int64_t n = L->last_nnz;
    bool ok = true;
    if (unique && U > 0) {
        widen_u32<<<grid_for(U, 256), 256, 0, st>>>(L->last_unique32, L->num_unique, U, unique);
        L->launches += 1;
    }
    if (inverse && n > 0)
        ok = ok && cudaMemcpyAsync(inverse, L->inverse, sizeof(int32_t) * n, cudaMemcpyDeviceToDevice, st) == cudaSuccess;
    if (counts && U > 0)
        ok = ok && cudaMemcpyAsync(counts, L->cnt, sizeof(int32_t) * U, cudaMemcpyDeviceToDevice, st) == cudaSuccess;
    if (seg_offsets)
        ok = ok && cudaMemcpyAsync(seg_offsets, L->seg_off, sizeof(int32_t) * (U + 1), cudaMemcpyDeviceToDevice, st) ==
                       cudaSuccess;
    if (sorted_bags && n > 0)
        ok = ok && cudaMemcpyAsync(sorted_bags, L->last_sorted_bags, sizeof(int32_t) * n, cudaMemcpyDeviceToDevice,
                                   st) == cudaSuccess;
    if (num_unique_host) *num_unique_host = U;
    if (!ok || cudaGetLastError() != cudaSuccess) return EMB_ERR_CUDA;
    return EMB_OK;
}

int emb_unique_workspace(int64_t n, size_t* bytes)
{
    if (!bytes || n < 0 || n >= (int64_t(1) << 31)) return EMB_ERR_INVALID_ARG;
    *bytes = unique_ws_layout(n, nullptr).total;
    return EMB_OK;
}

int emb_unique(const int64_t* keys, int64_t n, int64_t* unique, int32_t* inverse, int32_t* counts,
               int32_t* seg_offsets, int64_t* num_unique, void* workspace, size_t workspace_bytes, void* stream)
{
    if (!emb::unique_args_valid(keys, n, unique, inverse, counts, seg_offsets, num_unique)) return EMB_ERR_INVALID_ARG;
    UniqueWs w = unique_ws_layout(n, nullptr);
    if (!workspace || workspace_bytes < w.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return EMB_ERR_INVALID_ARG;
    w = unique_ws_layout(n, static_cast<char*>(workspace));
    cudaStream_t st = S(stream);
    int32_t* seg = seg_offsets ? seg_offsets : w.seg;
    if (n == 0) {
        if (cudaMemsetAsync(num_unique, 0, sizeof(int64_t), st) != cudaSuccess) return EMB_ERR_CUDA;
        if (cudaMemsetAsync(seg, 0, sizeof(int32_t), st) != cudaSuccess) return EMB_ERR_CUDA;
        return EMB_OK;
    }
    SortPlan plan = make_sort_plan(n, 64);
    if (launch_minmax(keys, n, w.mm, w.key_sub, w.bits, st) < 0) return EMB_ERR_CUDA;
    SortArgs sa = sort_args(keys, nullptr, w.k_out, w.v_out, w.k_tmp, w.v_tmp, n);
    sa.bits_dev = w.bits;
    sa.key_sub = w.key_sub;
    if (radix_sort_pairs<uint64_t>(plan, sa, w.sort_scratch, st) < 0) return EMB_ERR_CUDA;
    if (rle_sorted<uint64_t>(w.k_out, w.v_out, n, ~0ull, w.key_sub, unique, nullptr, seg, counts, inverse, num_unique,
                             w.rle, nullptr, st) < 0)
        return EMB_ERR_CUDA;
    return EMB_OK;
}

int emb_get_rows(emb_layer* L, int32_t t, int64_t row0, int64_t n, void* weights_host, float* state_host,
                 void* stream)
{
    if (!L || t < 0 || t >= L->T || row0 < 0 || n < 0 || row0 + n > L->tabs[t].rows || (n > 0 && !weights_host))
        return EMB_ERR_INVALID_ARG;
    const TableDev& d = L->tabs[t];
    if (state_host && !d.state) return EMB_ERR_INVALID_ARG;
    cudaStream_t st = S(stream);
    const size_t eb = dtype_bytes(d.dtype);
    bool ok = cudaMemcpyAsync(weights_host, static_cast<char*>(d.w) + (size_t)row0 * d.dim * eb,
                              (size_t)n * d.dim * eb, cudaMemcpyDeviceToHost, st) == cudaSuccess;
    if (ok && state_host)
        ok = cudaMemcpyAsync(state_host, d.state + (size_t)row0 * state_cols(d), sizeof(float) * (size_t)n * state_cols(d),
                             cudaMemcpyDeviceToHost, st) == cudaSuccess;
    ok = ok && cudaStreamSynchronize(st) == cudaSuccess;
    return ok ? EMB_OK : EMB_ERR_CUDA;
}

int emb_set_rows(emb_layer* L, int32_t t, int64_t row0, int64_t n, const void* weights_host, const float* state_host,
                 void* stream)
{
    if (!L || t < 0 || t >= L->T || row0 < 0 || n < 0 || row0 + n > L->tabs[t].rows || (n > 0 && !weights_host))
        return EMB_ERR_INVALID_ARG;
    const TableDev& d = L->tabs[t];
    if (state_host && !d.state) return EMB_ERR_INVALID_ARG;
    cudaStream_t st = S(stream);
    const size_t eb = dtype_bytes(d.dtype);
    bool ok = cudaMemcpyAsync(static_cast<char*>(d.w) + (size_t)row0 * d.dim * eb, weights_host,
                              (size_t)n * d.dim * eb, cudaMemcpyHostToDevice, st) == cudaSuccess;
    if (ok && state_host)
        ok = cudaMemcpyAsync(d.state + (size_t)row0 * state_cols(d), state_host, sizeof(float) * (size_t)n * state_cols(d),
                             cudaMemcpyHostToDevice, st) == cudaSuccess;
    ok = ok && cudaStreamSynchronize(st) == cudaSuccess;
    return ok ? EMB_OK : EMB_ERR_CUDA;
}

int emb_cache_build(emb_layer* L, int32_t t, const int64_t* rows, int64_t n, void* stream)
{
    if (!L || t < 0 || t >= L->T || n < 0 || n >= (int64_t(1) << 30) || (n > 0 && !rows) || !aligned_to(rows, 8) ||
        (n > 0 && L->tabs[t].rows >= (int64_t(1) << 31)))
        return EMB_ERR_INVALID_ARG;
    cudaStream_t st = S(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return EMB_ERR_CUDA;
    TableDev& d = L->tabs[t];
    auto& cb = L->cache_bufs[t];
    if (cb.first) cudaFree(cb.first);
    if (cb.second) cudaFree(cb.second);
    cb = std::make_pair(nullptr, nullptr);
    d.cache_w = nullptr;
    d.cache_map = nullptr;
    d.cache_mask = 0;
    int rc = EMB_OK;
    if (n > 0) {
        uint64_t cap = 64;
        while (cap < 2 * (uint64_t)n) cap <<= 1;
        void *w = nullptr, *m = nullptr;
        if (cudaMalloc(&w, sizeof(__half) * (size_t)n * d.dim) != cudaSuccess ||
            cudaMalloc(&m, sizeof(unsigned long long) * cap) != cudaSuccess) {
            cudaGetLastError();
            if (w) cudaFree(w);
            rc = EMB_ERR_OOM;
        } else {
            cb = std::make_pair(w, m);
            d.cache_mask = (uint32_t)(cap - 1);
            if (cudaMemsetAsync(m, 0xFF, sizeof(unsigned long long) * cap, st) != cudaSuccess) rc = EMB_ERR_CUDA;
            if (rc == EMB_OK)
                rc = track(L, launch_cache_fill(d, t, rows, n, static_cast<__half*>(w),
                                                static_cast<unsigned long long*>(m), d.cache_mask, L->err, st));
            d.cache_w = static_cast<const __half*>(w);
            d.cache_map = static_cast<const unsigned long long*>(m);
        }
    }
    if (cudaMemcpyAsync(L->d_tables + t, &d, sizeof(TableDev), cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        rc = EMB_ERR_CUDA;
    return rc;
}

int emb_forward_infer(emb_layer* L, const int64_t* keys, const int64_t* offsets, const int32_t* table_ids,
                      int64_t nnz, int32_t batch, float* out, void* stream)
{
    if (!L || !offsets || !table_ids || !out || batch < 1 || batch > L->max_batch || nnz < 0 || nnz > L->max_nnz ||
        (nnz > 0 && !keys) || !aligned16(out) || !aligned_to(keys, 8) || !aligned_to(offsets, 8) ||
        !aligned_to(table_ids, 4))
        return EMB_ERR_INVALID_ARG;
    cudaStream_t st = S(stream);
    // the side stream's dedup may still read the resolved rows rewritten here
    if (L->early_pending && cudaStreamWaitEvent(st, L->ev_ready, 0) != cudaSuccess) return EMB_ERR_CUDA;
    InferArgs ia;
    ia.keys = keys;
    ia.offsets = offsets;
    ia.nnz = nnz;
    ia.batch = batch;
    ia.tables = L->d_tables;
    ia.dyn_tables = L->d_dyn_tables;
    ia.num_dyn = L->num_dyn;
    ia.resolved = L->resolved;
    int rc = track(L, launch_infer_resolve(ia, nnz, st));
    if (rc != EMB_OK) return rc;
    FwdArgs a;
    a.keys = keys;
    a.offsets = offsets;
    a.nnz = nnz;
    a.table_ids = table_ids;
    a.batch = batch;
    a.num_tables = L->T;
    a.out = out;
    a.ld = L->total_dim;
    a.tables = L->d_tables;
    a.gid_out = nullptr;
    a.bag_out = nullptr;
    a.tab_start = nullptr;
    a.bag_scale = nullptr;
    a.sentinel = (uint32_t)L->total_rows;
    a.warps_per_table = (batch + 31) / 32;
    a.order_buf = L->table_order;
    a.write_ids = false;
    a.rows16 = true;
    for (const TableDev& d : L->tabs) a.rows16 = a.rows16 && d.dtype != EMB_F32;
    a.resolved = L->resolved;
    a.infer = true;
    a.err = L->err;
    return track(L, launch_forward(a, st));
}

int emb_find_keys(emb_layer* L, int32_t t, const int64_t* keys, int64_t n, int64_t* rows_out, void* stream)
{
    if (!L || t < 0 || t >= L->T || n < 0 || (n > 0 && (!keys || !rows_out)) || !L->tabs[t].dynamic ||
        !aligned_to(keys, 8) || !aligned_to(rows_out, 8))
        return EMB_ERR_INVALID_ARG;
    return track(L, launch_dyn_find(L->d_tables, t, keys, n, rows_out, S(stream)));
}

int emb_get_master_rows(emb_layer* L, int32_t t, int64_t row0, int64_t n, float* master_host, void* stream)
{
    if (!L || t < 0 || t >= L->T || row0 < 0 || n < 0 || row0 + n > L->tabs[t].rows || (n > 0 && !master_host) ||
        !L->tabs[t].master)
        return EMB_ERR_INVALID_ARG;
    const TableDev& d = L->tabs[t];
    cudaStream_t st = S(stream);
    const bool ok = cudaMemcpyAsync(master_host, d.master + (size_t)row0 * d.dim, sizeof(float) * (size_t)n * d.dim,
                                    cudaMemcpyDeviceToHost, st) == cudaSuccess &&
                    cudaStreamSynchronize(st) == cudaSuccess;
    return ok ? EMB_OK : EMB_ERR_CUDA;
}

int emb_set_master_rows(emb_layer* L, int32_t t, int64_t row0, int64_t n, const float* master_host, void* stream)
{
    if (!L || t < 0 || t >= L->T || row0 < 0 || n < 0 || row0 + n > L->tabs[t].rows || (n > 0 && !master_host) ||
        !L->tabs[t].master)
        return EMB_ERR_INVALID_ARG;
    const TableDev& d = L->tabs[t];
    cudaStream_t st = S(stream);
    const bool ok = cudaMemcpyAsync(d.master + (size_t)row0 * d.dim, master_host, sizeof(float) * (size_t)n * d.dim,
                                    cudaMemcpyHostToDevice, st) == cudaSuccess &&
                    cudaStreamSynchronize(st) == cudaSuccess;
    return ok ? EMB_OK : EMB_ERR_CUDA;
}

int emb_gather_master_rows(emb_layer* L, int32_t t, const int64_t* rows, int64_t n, float* master_out, void* stream)
{
    if (!L || t < 0 || t >= L->T || n < 0 || (n > 0 && (!rows || !master_out)) || !L->tabs[t].master ||
        !aligned_to(rows, 8) || !aligned_to(master_out, 4))
        return EMB_ERR_INVALID_ARG;
    if (n == 0) return EMB_OK;
    const TableDev& d = L->tabs[t];
    gather_rows_kernel<<<grid_for(n * d.dim, 256), 256, 0, S(stream)>>>(d.master, nullptr, 0, EMB_F32, d.rows, d.dim,
                                                                        rows, n, master_out, nullptr, L->err);
    L->launches += 1;
    return cudaGetLastError() == cudaSuccess ? EMB_OK : EMB_ERR_CUDA;
}

int emb_gather_rows(emb_layer* L, int32_t t, const int64_t* rows, int64_t n, void* weights_out, float* state_out,
                    void* stream)
{
    if (!L || t < 0 || t >= L->T || n < 0 || (n > 0 && (!rows || !weights_out))) return EMB_ERR_INVALID_ARG;
    const TableDev& d = L->tabs[t];
    if (!aligned_to(rows, 8) || !aligned_to(weights_out, dtype_bytes(d.dtype)) || !aligned_to(state_out, 4))
        return EMB_ERR_INVALID_ARG;
    if (state_out && !d.state) return EMB_ERR_INVALID_ARG;
    if (n == 0) return EMB_OK;
    gather_rows_kernel<<<grid_for(n * d.dim, 256), 256, 0, S(stream)>>>(
        d.w, d.state, (int)state_cols(d), d.dtype, d.rows, d.dim, rows, n, weights_out, state_out, L->err);
    L->launches += 1;
    return cudaGetLastError() == cudaSuccess ? EMB_OK : EMB_ERR_CUDA;
}

int emb_sync_status(emb_layer* L, void* stream)
{
    if (!L) return EMB_ERR_INVALID_ARG;
    cudaStream_t st = S(stream);
    int bits = 0;
    if (cudaMemcpyAsync(&bits, L->err, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess || cudaMemsetAsync(L->err, 0, sizeof(int), st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return EMB_ERR_CUDA;
    if (bits & ERRBIT_CAPACITY) return EMB_ERR_CAPACITY;
    if (bits & ERRBIT_KEY_RANGE) return EMB_ERR_KEY_RANGE;
    if (bits & (ERRBIT_TABLE_ID | ERRBIT_OFFSETS)) return EMB_ERR_INVALID_ARG;
    if (bits & ERRBIT_TIMEOUT) return EMB_ERR_TIMEOUT;
    return EMB_OK;
}

int emb_set_timing(emb_layer* L, int32_t enable)
{
    if (!L) return EMB_ERR_INVALID_ARG;
    if (enable && !L->tslot[0].ev[0]) {
        for (auto& s : L->tslot)
            for (cudaEvent_t& e : s.ev)
                if (cudaEventCreate(&e) != cudaSuccess) return EMB_ERR_CUDA;
    }
    if (!enable) harvest_timing(L);
    L->timing = enable != 0;
    return EMB_OK;
}

int emb_phase_times(emb_layer* L, float* ms_host, int32_t n, int64_t* steps_host, int32_t reset)
{
    if (!L || n < 0 || n > EMB_NUM_PHASES || (n > 0 && !ms_host)) return EMB_ERR_INVALID_ARG;
    harvest_timing(L);
    for (int i = 0; i < n; ++i) ms_host[i] = (float)L->phase_ms[i];
    if (steps_host) *steps_host = L->timed_steps;
    if (reset) {
        for (double& v : L->phase_ms) v = 0.0;
        L->timed_steps = 0;
    }
    return EMB_OK;
}

int emb_launch_count(emb_layer* L, int64_t* count_host, int32_t reset)
{
    if (!L || !count_host) return EMB_ERR_INVALID_ARG;
    *count_host = L->launches;
    if (reset) L->launches = 0;
    return EMB_OK;
}

}  // extern "C"
