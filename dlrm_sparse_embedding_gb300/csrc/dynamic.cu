// Dynamic tables: arbitrary int64 keys mapped to rows by a GPU hash map with
// insert on first lookup -- the GPU hash table behind HugeCTR's embedding
// (GTC 2022 "Merlin HugeCTR" slides, "HUGECTR EMBEDDING LAYER") without
// eviction.
//
// The map is open addressing over the table's own rows: map_keys[r] is the
// key that owns row r (kMapEmpty when free), so a key's slot is its row and
// nothing downstream of the forward changes.  A key is placed by linear
// probing from a fixed hash of (table, key).  The thread whose compare-and-
// swap claims a free row writes that row's initial values (the counter-based
// generator of emb_init_uniform, keyed by the key instead of the row), its
// Adagrad state and its fp32 master; other lookups of the key in the same
// launch only read the row index, and the rows themselves are read by later
// kernels.  Probing is bounded by the table's rows; a full table reports
// ERRBIT_CAPACITY and the lookup is skipped.  No thread waits on another.
#include "emb_internal.cuh"

namespace emb {

namespace {

__device__ __forceinline__ uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// First probe position of `key` in a map of `rows` rows.
__device__ __forceinline__ int64_t home_row(uint64_t key, int t, int64_t rows)
{
    const uint64_t h = mix64(key + 0x9E3779B97F4A7C15ull * (uint64_t)(t + 1));
    return (int64_t)__umul64hi(h, (uint64_t)rows);
}

// Initial values of the row taken by `key` in table t: column c gets
// lo + (hi - lo) * ((h >> 40) * 2^-24) with h splitmix64 output number
// (key << 8) ^ (t << 57) ^ c of the stream started from `seed`, in fp32.
__device__ void init_row(const DynArgs& a, const TableDev& tb, int t, uint64_t key, int64_t row)
{
    const float d = __fsub_rn(a.hi, a.lo);
    const int64_t e0 = row * tb.dim;
    for (int c = 0; c < tb.dim; ++c) {
        const uint64_t n = (key << 8) ^ ((uint64_t)t << 57) ^ (uint64_t)c;
        const uint64_t z = mix64(a.seed + (n + 1ull) * 0x9E3779B97F4A7C15ull);
        const float f = __fmul_rn(__uint2float_rn((uint32_t)(z >> 40)), 5.9604644775390625e-08f);
        const float v = __fadd_rn(a.lo, __fmul_rn(d, f));
        if (tb.dtype == EMB_F32) static_cast<float*>(tb.w)[e0 + c] = v;
        else if (tb.dtype == EMB_F16) static_cast<__half*>(tb.w)[e0 + c] = __float2half_rn(v);
        else static_cast<__nv_bfloat16*>(tb.w)[e0 + c] = __float2bfloat16_rn(v);
        if (tb.master) tb.master[e0 + c] = v;
        if (tb.opt == EMB_OPT_ADAGRAD) tb.state[e0 + c] = a.init_acc[t];
    }
    if (tb.opt == EMB_OPT_ROWWISE_ADAGRAD) tb.state[row] = a.init_acc[t];
}

// Grid (x, dynamic table): threads stride over the table's lookups.
__global__ void dyn_resolve(DynArgs a)
{
    const int t = a.dyn_tables[blockIdx.y];
    const TableDev& tb = a.tables[t];
    const int64_t p0 = clamp_offset(a.offsets[(int64_t)t * a.batch], 0, a.nnz);
    const int64_t p1 = clamp_offset(a.offsets[(int64_t)(t + 1) * a.batch], p0, a.nnz);
    for (int64_t i = p0 + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < p1;
         i += (int64_t)gridDim.x * blockDim.x) {
        const uint64_t key = (uint64_t)a.keys[i];
        int64_t row = -1;
        if (key != kMapEmpty) {
            int64_t s = home_row(key, t, tb.rows);
            for (int64_t probe = 0; probe < tb.rows; ++probe) {
                const unsigned long long cur = tb.map_keys[s];
                if (cur == key) {
                    row = s;
                    break;
                }
                if (cur == kMapEmpty) {
                    const unsigned long long prev = atomicCAS(tb.map_keys + s, kMapEmpty, key);
                    if (prev == kMapEmpty) {
                        row = s;
                        init_row(a, tb, t, key, s);
                        break;
                    }
                    if (prev == key) {
                        row = s;
                        break;
                    }
                }
                if (++s == tb.rows) s = 0;
            }
            if (row < 0) atomicOr(a.err, ERRBIT_CAPACITY);
        }
        a.resolved[i] = row;
    }
}

__global__ void dyn_find(const TableDev* __restrict__ tables, int t, const int64_t* __restrict__ keys, int64_t n,
                         int64_t* __restrict__ rows_out)
{
    const TableDev& tb = tables[t];
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const uint64_t key = (uint64_t)keys[i];
        int64_t row = -1;
        if (key != kMapEmpty) {
            int64_t s = home_row(key, t, tb.rows);
            for (int64_t probe = 0; probe < tb.rows; ++probe) {
                const unsigned long long cur = tb.map_keys[s];
                if (cur == key) {
                    row = s;
                    break;
                }
                if (cur == kMapEmpty) break;
                if (++s == tb.rows) s = 0;
            }
        }
        rows_out[i] = row;
    }
}

__global__ void dyn_clear(unsigned long long* map_keys, int64_t rows)
{
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < rows; i += (int64_t)gridDim.x * blockDim.x)
        map_keys[i] = kMapEmpty;
}

unsigned grid_of(int64_t n, int threads, int64_t cap)
{
    int64_t b = (n + threads - 1) / threads;
    if (b < 1) b = 1;
    if (b > cap) b = cap;
    return (unsigned)b;
}

}  // namespace

int launch_dyn_resolve(const DynArgs& a, int64_t nnz, cudaStream_t st)
{
    if (a.num_dyn <= 0 || nnz <= 0) return 0;
    // enough blocks per table for its share of lookups; threads stride over the rest
    const unsigned gx = grid_of(nnz / a.num_dyn + 1, 256, 4096);
    dyn_resolve<<<dim3(gx, (unsigned)a.num_dyn), 256, 0, st>>>(a);
    return cudaGetLastError() == cudaSuccess ? 1 : -1;
}

int launch_dyn_find(const TableDev* tables, int t, const int64_t* keys, int64_t n, int64_t* rows_out, cudaStream_t st)
{
    if (n <= 0) return 0;
    dyn_find<<<grid_of(n, 256, 4096), 256, 0, st>>>(tables, t, keys, n, rows_out);
    return cudaGetLastError() == cudaSuccess ? 1 : -1;
}

int launch_dyn_clear(unsigned long long* map_keys, int64_t rows, cudaStream_t st)
{
    if (rows <= 0) return 0;
    dyn_clear<<<grid_of(rows, 256, 65536), 256, 0, st>>>(map_keys, rows);
    return cudaGetLastError() == cudaSuccess ? 1 : -1;
}

}  // namespace emb
