// Inference-only forward with fp16 caches of hot rows.
//
// The GTC 2022 "Merlin HugeCTR" slides (slide "HUGECTR: SCALABLE, ACCELERATED
// RECSYS TRAINING") serve inference through an embedding cache on the GPU in
// front of a hierarchical parameter server (HPS).  Here a table
// may hold a cache of chosen rows as fp16 copies (half the bytes of an fp32
// row, so a hot set stays in L2); the inference forward reads a cached row
// from the cache and every other row from the table.  The cache is a snapshot
// taken when it is built: later training steps do not refresh it.
//
// The pooling is the training forward's kernel (fwd_pool) instantiated for
// inference: the lane that loads a key also looks its row up in the table's
// cache map (open addressing of (row, slot) pairs) and reads a cached row from
// the fp16 cache; no ids or bag scales are written, so a following backward
// still refers to the last training forward.  Dynamic tables first find their
// keys' rows without inserting (infer_resolve).
#include "emb_internal.cuh"

namespace emb {

namespace {

__device__ __forceinline__ uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// first probe of `row` in a cache map
__device__ __forceinline__ uint32_t cache_home(uint64_t row) { return (uint32_t)mix64(row + 0x632BE59BD9B4E019ull); }

__global__ void cache_fill(TableDev tb, const int64_t* __restrict__ rows, int64_t n, __half* __restrict__ cache_w,
                           unsigned long long* __restrict__ cache_map, uint32_t mask, int* err)
{
    const int dim = tb.dim;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = rows[i];
        if (r < 0 || r >= tb.rows) {
            atomicOr(err, ERRBIT_KEY_RANGE);
            continue;
        }
        const unsigned long long entry = ((unsigned long long)r << 32) | (unsigned long long)i;
        uint32_t s = cache_home((uint64_t)r) & mask;
        bool mine = false;
        for (uint32_t probe = 0; probe <= mask; ++probe) {
            const unsigned long long prev = atomicCAS(cache_map + s, kCacheEmpty, entry);
            if (prev == kCacheEmpty) {
                mine = true;
                break;
            }
            if ((prev >> 32) == (unsigned long long)r) break;   // held already: the earlier slot stays
            s = (s + 1) & mask;
        }
        if (!mine) continue;
        for (int c = 0; c < dim; ++c) {
            float v;
            const int64_t e = r * dim + c;
            if (tb.dtype == EMB_F32) v = static_cast<const float*>(tb.w)[e];
            else if (tb.dtype == EMB_F16) v = __half2float(static_cast<const __half*>(tb.w)[e]);
            else v = __bfloat162float(static_cast<const __nv_bfloat16*>(tb.w)[e]);
            cache_w[i * dim + c] = __float2half_rn(v);
        }
    }
}

// Grid (x, dynamic table): the row of every lookup of the table, found
// without inserting (-1 for an id the table never saw).
__global__ void infer_resolve(InferArgs a)
{
    const int t = a.dyn_tables[blockIdx.y];
    const TableDev& tb = a.tables[t];
    const int64_t p0 = clamp_offset(a.offsets[(int64_t)t * a.batch], 0, a.nnz);
    const int64_t p1 = clamp_offset(a.offsets[(int64_t)(t + 1) * a.batch], p0, a.nnz);
    for (int64_t i = p0 + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < p1;
         i += (int64_t)gridDim.x * blockDim.x) {
        const uint64_t k = (uint64_t)a.keys[i];
        int64_t row = -1;
        if (k != kMapEmpty) {
            const uint64_t h = mix64(k + 0x9E3779B97F4A7C15ull * (uint64_t)(t + 1));
            int64_t s = (int64_t)__umul64hi(h, (uint64_t)tb.rows);
            for (int64_t probe = 0; probe < tb.rows; ++probe) {
                const unsigned long long cur = tb.map_keys[s];
                if (cur == k) {
                    row = s;
                    break;
                }
                if (cur == kMapEmpty) break;
                if (++s == tb.rows) s = 0;
            }
        }
        a.resolved[i] = row;
    }
}

unsigned grid_of(int64_t n, int threads, int64_t cap)
{
    int64_t b = (n + threads - 1) / threads;
    if (b < 1) b = 1;
    if (b > cap) b = cap;
    return (unsigned)b;
}

}  // namespace

int launch_cache_fill(const TableDev& tb, int t, const int64_t* rows, int64_t n, __half* cache_w,
                      unsigned long long* cache_map, uint32_t cache_mask, int* err, cudaStream_t st)
{
    (void)t;
    if (n <= 0) return 0;
    cache_fill<<<grid_of(n, 256, 4096), 256, 0, st>>>(tb, rows, n, cache_w, cache_map, cache_mask, err);
    return cudaGetLastError() == cudaSuccess ? 1 : -1;
}

int launch_infer_resolve(const InferArgs& a, int64_t nnz, cudaStream_t st)
{
    if (nnz <= 0 || a.num_dyn <= 0) return 0;
    const unsigned gx = grid_of(nnz / a.num_dyn + 1, 256, 4096);
    infer_resolve<<<dim3(gx, (unsigned)a.num_dyn), 256, 0, st>>>(a);
    return cudaGetLastError() == cudaSuccess ? 1 : -1;
}

}  // namespace emb
