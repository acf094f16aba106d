// Dedup helpers of the unique-based backward and of emb_unique.
//
// Hash-based unique (the UB flavour of "NVIDIA EMBark revoluciona la formacion
// en sistemas de recomendacion a escala", section "Integracion del cluster";
// the GPU hash table of the GTC 2022 HugeCTR slide "HUGECTR EMBEDDING
// LAYER"): every lookup's global row id goes into an open-addressing table
// (linear probing, bounded by the capacity, no waits); each newly inserted id
// is appended to a compact list with one global atomic per block.  Only that
// short list is then sorted, which gives the canonical ascending order, the
// rank of every slot and so the inverse index of every lookup.
#include "emb_internal.cuh"

namespace emb {

namespace {

__device__ __forceinline__ uint32_t mix32(uint32_t h)
{
    // murmur3 32-bit finaliser
    h ^= h >> 16;
    h *= 0x85ebca6bu;
    h ^= h >> 13;
    h *= 0xc2b2ae35u;
    h ^= h >> 16;
    return h;
}

constexpr int kHashThreads = 256;

__global__ void __launch_bounds__(kHashThreads)
hash_insert(const uint32_t* __restrict__ gid, int64_t n, uint32_t limit, uint32_t* table, uint32_t mask,
            uint32_t* __restrict__ slot_of, uint32_t* __restrict__ ukey, uint32_t* __restrict__ uslot,
            int64_t* ucount, int* err)
{
    __shared__ uint32_t s_cnt;
    __shared__ unsigned long long s_base;
    __shared__ uint32_t s_key[kHashThreads], s_slot[kHashThreads];
    if (threadIdx.x == 0) s_cnt = 0;
    __syncthreads();
    const int64_t i = (int64_t)blockIdx.x * kHashThreads + threadIdx.x;
    bool fresh = false;
    uint32_t slot = kNoSlot, g = 0;
    if (i < n) {
        g = gid[i];
        if (g < limit) {
            uint32_t s = mix32(g) & mask;
            for (uint32_t probe = 0; probe <= mask; ++probe) {
                uint32_t cur = __ldcg(table + s);
                if (cur == g) { slot = s; break; }
                if (cur == kEmptySlot) {
                    uint32_t prev = atomicCAS(table + s, kEmptySlot, g);
                    if (prev == kEmptySlot) { slot = s; fresh = true; break; }
                    if (prev == g) { slot = s; break; }
                }
                s = (s + 1) & mask;
            }
            if (slot == kNoSlot) atomicOr(err, ERRBIT_CAPACITY);
        }
        slot_of[i] = slot;
    }
    uint32_t li = 0;
    if (fresh) li = atomicAdd(&s_cnt, 1u);
    __syncthreads();
    if (threadIdx.x == 0 && s_cnt) s_base = atomicAdd(reinterpret_cast<unsigned long long*>(ucount),
                                                      (unsigned long long)s_cnt);
    __syncthreads();
    if (fresh) {
        s_key[li] = g;
        s_slot[li] = slot;
    }
    __syncthreads();
    if (threadIdx.x < s_cnt) {
        ukey[s_base + threadIdx.x] = s_key[threadIdx.x];
        uslot[s_base + threadIdx.x] = s_slot[threadIdx.x];
    }
}

// rank of every used slot; bits needed to sort values 0..U; seg_off[U] = n.
__global__ void hash_rank(const uint32_t* __restrict__ sslot, const int64_t* __restrict__ U_dev,
                          uint32_t* __restrict__ slot_rank, int32_t* bits_dev, int32_t* seg_off, int64_t n)
{
    const int64_t U = *U_dev;
    const int64_t r0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (r0 == 0) {
        *bits_dev = 32 - __clz((uint32_t)U);
        seg_off[U] = (int32_t)n;
    }
    for (int64_t r = r0; r < U; r += (int64_t)gridDim.x * blockDim.x) slot_rank[sslot[r]] = (uint32_t)r;
}

__global__ void hash_inverse(const uint32_t* __restrict__ slot_of, int64_t n, const uint32_t* __restrict__ slot_rank,
                             const int64_t* __restrict__ U_dev, uint32_t* __restrict__ inv)
{
    const uint32_t U = (uint32_t)*U_dev;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const uint32_t s = slot_of[i];
        inv[i] = s == kNoSlot ? U : __ldg(slot_rank + s);
    }
}

// seg_off from lookups sorted by inverse index (keys >= U are skipped lookups).
__global__ void seg_from_sorted(const uint32_t* __restrict__ sk, int64_t n, const int64_t* __restrict__ U_dev,
                                int32_t* __restrict__ seg_off)
{
    const uint32_t U = (uint32_t)*U_dev;
    for (int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; p < n; p += (int64_t)gridDim.x * blockDim.x) {
        const uint32_t k = sk[p];
        const uint32_t kp = p > 0 ? sk[p - 1] : 0xFFFFFFFFu;
        if (k < U) {
            if (p == 0 || kp != k) seg_off[k] = (int32_t)p;
        } else if (p == 0 || kp < U) {
            seg_off[U] = (int32_t)p;
        }
    }
}

__global__ void hash_clear(uint32_t* table, const uint32_t* __restrict__ sslot, const int64_t* __restrict__ U_dev)
{
    const int64_t U = *U_dev;
    for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < U; r += (int64_t)gridDim.x * blockDim.x)
        table[sslot[r]] = kEmptySlot;
}

__global__ void gather_u32(const uint32_t* __restrict__ src, const uint32_t* __restrict__ idx, int64_t n,
                           uint32_t* __restrict__ dst)
{
    for (int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; p < n; p += (int64_t)gridDim.x * blockDim.x)
        dst[p] = src[idx[p]];
}

__global__ void counts_from_offsets(const int32_t* __restrict__ seg_off, const int64_t* __restrict__ U_dev,
                                    int64_t n_max, int32_t* __restrict__ counts)
{
    const int64_t U = *U_dev;
    for (int64_t s = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; s < U && s < n_max;
         s += (int64_t)gridDim.x * blockDim.x)
        counts[s] = seg_off[s + 1] - seg_off[s];
}

__global__ void minmax_init(unsigned long long* mm)
{
    mm[0] = 0xFFFFFFFFFFFFFFFFull;   // min of biased keys
    mm[1] = 0ull;                    // max of biased keys
}

// keys are compared as int64; store them biased (x ^ 2^63) so unsigned atomics order them.
__global__ void minmax_keys(const int64_t* __restrict__ keys, int64_t n, unsigned long long* mm)
{
    unsigned long long lo = 0xFFFFFFFFFFFFFFFFull, hi = 0ull;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        unsigned long long b = (unsigned long long)keys[i] ^ 0x8000000000000000ull;
        lo = b < lo ? b : lo;
        hi = b > hi ? b : hi;
    }
    for (int o = 16; o > 0; o >>= 1) {
        unsigned long long l2 = __shfl_xor_sync(0xffffffffu, lo, o), h2 = __shfl_xor_sync(0xffffffffu, hi, o);
        lo = l2 < lo ? l2 : lo;
        hi = h2 > hi ? h2 : hi;
    }
    if ((threadIdx.x & 31) == 0) {
        atomicMin(mm, lo);
        atomicMax(mm + 1, hi);
    }
}

// min key (as the value to subtract from every key) and the bits of max-min.
__global__ void minmax_finish(const unsigned long long* mm, uint64_t* key_sub, int32_t* bits_dev)
{
    const unsigned long long lo = mm[0] ^ 0x8000000000000000ull, hi = mm[1] ^ 0x8000000000000000ull;
    *key_sub = lo;
    const unsigned long long range = hi - lo;
    *bits_dev = range ? 64 - __clzll((long long)range) : 1;
}

inline unsigned grid_for(int64_t n, int threads, int cap = 8192)
{
    int64_t b = (n + threads - 1) / threads;
    if (b < 1) b = 1;
    if (b > cap) b = cap;
    return (unsigned)b;
}

}  // namespace

// ---------------------------------------------------------------------------
// launchers (each returns kernels launched, or -1)
// ---------------------------------------------------------------------------

int launch_hash_insert(const uint32_t* gid, int64_t n, uint32_t limit, uint32_t* table, uint32_t mask,
                       uint32_t* slot_of, uint32_t* ukey, uint32_t* uslot, int64_t* ucount, int* err,
                       cudaStream_t st)
{
    if (cudaMemsetAsync(ucount, 0, sizeof(int64_t), st) != cudaSuccess) return -1;
    if (n <= 0) return 0;
    hash_insert<<<(unsigned)((n + kHashThreads - 1) / kHashThreads), kHashThreads, 0, st>>>(
        gid, n, limit, table, mask, slot_of, ukey, uslot, ucount, err);
    return cudaGetLastError() == cudaSuccess ? 1 : -1;
}

int launch_hash_rank_inverse(const uint32_t* sslot, const int64_t* U_dev, uint32_t* slot_rank, int32_t* bits_dev,
                             int32_t* seg_off, const uint32_t* slot_of, int64_t n, uint32_t* inv, cudaStream_t st)
{
    hash_rank<<<grid_for(n, 256), 256, 0, st>>>(sslot, U_dev, slot_rank, bits_dev, seg_off, n);
    hash_inverse<<<grid_for(n, 256), 256, 0, st>>>(slot_of, n, slot_rank, U_dev, inv);
    return cudaGetLastError() == cudaSuccess ? 2 : -1;
}

int launch_seg_from_sorted(const uint32_t* sk, int64_t n, const int64_t* U_dev, int32_t* seg_off, int32_t* counts,
                           cudaStream_t st)
{
    if (n <= 0) return 0;
    seg_from_sorted<<<grid_for(n, 256), 256, 0, st>>>(sk, n, U_dev, seg_off);
    counts_from_offsets<<<grid_for(n, 256), 256, 0, st>>>(seg_off, U_dev, n, counts);
    return cudaGetLastError() == cudaSuccess ? 2 : -1;
}

int launch_hash_clear(uint32_t* table, const uint32_t* sslot, const int64_t* U_dev, int64_t n_max, cudaStream_t st)
{
    hash_clear<<<grid_for(n_max, 256), 256, 0, st>>>(table, sslot, U_dev);
    return cudaGetLastError() == cudaSuccess ? 1 : -1;
}

int launch_gather_u32(const uint32_t* src, const uint32_t* idx, int64_t n, uint32_t* dst, cudaStream_t st)
{
    if (n <= 0) return 0;
    gather_u32<<<grid_for(n, 256), 256, 0, st>>>(src, idx, n, dst);
    return cudaGetLastError() == cudaSuccess ? 1 : -1;
}

int launch_minmax(const int64_t* keys, int64_t n, unsigned long long* mm, uint64_t* key_sub, int32_t* bits_dev,
                  cudaStream_t st)
{
    minmax_init<<<1, 1, 0, st>>>(mm);
    minmax_keys<<<grid_for(n, 256, 2048), 256, 0, st>>>(keys, n, mm);
    minmax_finish<<<1, 1, 0, st>>>(mm, key_sub, bits_dev);
    return cudaGetLastError() == cudaSuccess ? 3 : -1;
}

}  // namespace emb
