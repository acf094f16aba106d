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
#include "reduce_chunks.cuh"

namespace emb {

namespace {

constexpr int kCombineThreads = 1024;   // combine block: all warps on a long row, or 4 groups of 256 on short ones
constexpr int kCombineGroups = 4;
constexpr int kCombineBlocksPerSM = 1;   // one 1024-thread block per SM
constexpr int kLongSegs = 32;            // blocks sharing one long split run ...
constexpr int kSegPieces = 1024;         // ... each adding at least this many of its pieces

// Barrier over `nthr` threads (a multiple of 32) on named barrier `bar`,
// returning how many of them passed pred.
__device__ __forceinline__ int group_count(int bar, int nthr, bool pred)
{
    int r;
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.popc.u32 %0, %2, %3, p;\n\t}"
                 : "=r"(r) : "r"((int)pred), "r"(bar), "r"(nthr) : "memory");
    return r;
}

__device__ __forceinline__ void group_sync(int bar, int nthr)
{
    asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(nthr) : "memory");
}

// Piece q of the split run whose first boundary is c: the tail piece of chunk
// c-1 (q = 0), then the head pieces of chunks c, c+1, ...
__device__ __forceinline__ const float* piece_ptr(const ReduceArgs& a, int64_t c, int64_t q)
{
    return q == 0 ? slot_ptr(a.slots, c - 1, kSlotTail) : slot_ptr(a.slots, c - 1 + q, kSlotHead);
}

// Compensated sum of pieces q0 .. q1-1 of the split run at boundary c over a
// group of nthr threads (tid its thread index, warps w0 .. w0 + nthr/32 - 1 of
// the block, named barrier bar): warp w adds pieces q0+w, q0+w+W, ... (four
// loads in flight), then the group's first warp adds the warps' sums in warp
// order; its lanes return the sum of their 4 columns in g.
__device__ __forceinline__ void sum_pieces(const ReduceArgs& a, int64_t c, int64_t q0, int64_t q1, bool colok,
                                           float (*part)[kMaxDim], int bar, int nthr, int tid, int w0, float g[4])
{
    const int W = nthr / 32;
    const int lane = tid & 31, warp = tid >> 5;
    float s[4] = {0.f, 0.f, 0.f, 0.f}, cc4[4] = {0.f, 0.f, 0.f, 0.f};
    if (colok) {
        int64_t qi = q0 + warp;
        for (; qi + 3 * W < q1; qi += 4 * W) {
            float4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) v[u] = *reinterpret_cast<const float4*>(piece_ptr(a, c, qi + u * W) + 4 * lane);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                kahan_add(s[0], cc4[0], v[u].x);
                kahan_add(s[1], cc4[1], v[u].y);
                kahan_add(s[2], cc4[2], v[u].z);
                kahan_add(s[3], cc4[3], v[u].w);
            }
        }
        for (; qi < q1; qi += W) {
            const float4 v = *reinterpret_cast<const float4*>(piece_ptr(a, c, qi) + 4 * lane);
            kahan_add(s[0], cc4[0], v.x);
            kahan_add(s[1], cc4[1], v.y);
            kahan_add(s[2], cc4[2], v.z);
            kahan_add(s[3], cc4[3], v.w);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) part[w0 + warp][4 * lane + q] = __fsub_rn(s[q], cc4[q]);
    }
    group_sync(bar, nthr);
    if (warp == 0) {
        float gs[4] = {0.f, 0.f, 0.f, 0.f}, gc[4] = {0.f, 0.f, 0.f, 0.f};
        if (colok) {
            for (int w = 0; w < W; ++w) {
#pragma unroll
                for (int q = 0; q < 4; ++q) kahan_add(gs[q], gc[q], part[w0 + w][4 * lane + q]);
            }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) g[q] = __fsub_rn(gs[q], gc[q]);
    }
}

// One warp applies the update of row `key` of table tb with gradient g (its
// lanes' 4 columns each).
__device__ __forceinline__ void apply_row(const ReduceArgs& a, const TableDev& tb, uint32_t key, const float g[4],
                                          int lane, bool colok)
{
    const float ssq = tb.opt == EMB_OPT_ROWWISE_ADAGRAD ? group_sum(sq4(g), 32, 0xffffffffu) : 0.f;
    const uint32_t gid = a.gid_of_key ? a.gid_of_key[key] : key;
    const int64_t row = (int64_t)gid - (int64_t)tb.row_base;
    // a row outside its table only comes from ids of a forward whose offsets were flagged
    if (colok && row >= 0 && row < tb.rows) {
        const int64_t elem = row * tb.dim + 4 * lane;
        apply_update4(tb, row, elem, g, load_update_w4(tb, elem), load_state4(tb, row, elem), ssq, lane == 0);
    }
}

// Chunk cc+1 starts inside the run of `key` iff the whole window of its
// nominal start holds the key (otherwise its start snapped to a later run).
__device__ __forceinline__ bool next_chunk_continues(const ReduceArgs& a, int64_t cc, uint32_t key)
{
    if (cc + 1 >= a.nchunks) return false;
    const int64_t win0 = (cc + 1) * a.chunk;
    const int64_t win1 = win0 + a.chunk < a.n ? win0 + a.chunk : a.n;
    return a.skeys[win0] == key && a.skeys[win1 - 1] == key;
}

// Adds the pieces of the split run that crosses boundary c (c*chunk), which
// starts in chunk c-1, and applies its update (a group as in sum_pieces).
__device__ __forceinline__ void combine_run(const ReduceArgs& a, int64_t c, int64_t& s_last, float (*part)[kMaxDim],
                                            int bar, int nthr, int tid, int w0)
{
    const int64_t pb = c * a.chunk;
    const uint32_t key = a.skeys[pb];
    for (int64_t base = c;; base += nthr) {
        const int cnt = group_count(bar, nthr, next_chunk_continues(a, base + tid, key));
        if (cnt < nthr) {
            if (tid == 0) s_last = base + cnt;
            break;
        }
    }
    group_sync(bar, nthr);
    const int64_t P = s_last - c + 2;   // tail piece of chunk c-1, head pieces of chunks c..last
    const uint32_t bag0 = a.sbags[pb];
    const int t = min((int)(bag0 / (uint32_t)a.batch), a.num_tables - 1);
    const TableDev tb = a.tables[t];
    const int lane = tid & 31;
    const bool colok = 4 * lane < tb.dim;
    float g[4];
    sum_pieces(a, c, 0, P, colok, part, bar, nthr, tid, w0, g);
    if ((tid >> 5) == 0) apply_row(a, tb, key, g, lane, colok);
}

// Segment `seg` of the long split run registered as long item `item`, by the
// whole block.  The run's pieces are cut into nseg = min(kLongSegs,
// max(1, P / kSegPieces)) equal ranges, each summed by one block (one segment:
// the block applies the update at once); otherwise the block
// that finishes a run's last outstanding segment (a counter per item, reset
// by that block) adds the segment sums in segment order and applies the
// update.  The run's extent comes from a kCombineThreads-ary search over the
// chunks (monotone: chunks continue the run, then stop).  No block waits on
// another.
__device__ __forceinline__ void combine_long_segment(const ReduceArgs& a, int item, int seg, float (*part)[kMaxDim],
                                                     int* s_flag)
{
    constexpr int T = kCombineThreads;
    const int tid = threadIdx.x, lane = tid & 31;
    const int64_t c = (int64_t)a.split_list[a.nchunks - 1 - item] + 1;
    const int64_t pb = c * a.chunk;
    const uint32_t key = a.skeys[pb];
    // segment seg exists only if the run has (seg + 1) * kSegPieces pieces or
    // more, i.e. it still continues past chunk c + (seg + 1) * kSegPieces - 3:
    // one probe spares the search for the segments a shorter run does not have
    if (seg > 0) {
        if (tid == 0) {
            *s_flag = next_chunk_continues(a, c + (int64_t)(seg + 1) * kSegPieces - 3, key);
            // the run's later segments do not exist either: the work counter skips them
            if (!*s_flag) atomicMax(a.split_count + 2, (item + 1) * kLongSegs);
        }
        group_sync(0, T);
        if (!*s_flag) return;
    }
    // last = the first chunk cc >= c whose next chunk does not continue the run
    int64_t lo = c, hi = a.nchunks - 1;
    while (lo < hi) {
        const int64_t step = (hi - lo + T - 1) / T;
        const int64_t x = lo + (int64_t)tid * step;
        const int cnt = group_count(0, T, x < hi && next_chunk_continues(a, x, key));
        const int64_t xc = lo + (int64_t)cnt * step;
        lo = cnt == 0 ? lo : lo + (int64_t)(cnt - 1) * step + 1;
        hi = xc < hi ? xc : hi;
    }
    const int64_t P = lo - c + 2;
    const int nseg = (int)min((int64_t)kLongSegs, max((int64_t)1, P / kSegPieces));
    if (seg >= nseg) return;
    const uint32_t bag0 = a.sbags[pb];
    const int t = min((int)(bag0 / (uint32_t)a.batch), a.num_tables - 1);
    const TableDev tb = a.tables[t];
    const bool colok = 4 * lane < tb.dim;
    const int64_t q0 = (int64_t)seg * P / nseg, q1 = (int64_t)(seg + 1) * P / nseg;
    float g[4];
    sum_pieces(a, c, q0, q1, colok, part, 0, T, tid, 0, g);
    if (nseg == 1) {   // the whole run in one segment
        if (tid < 32) apply_row(a, tb, key, g, lane, colok);
        return;
    }
    // the segment's sum replaces its first piece, which only this block read
    if (tid < 32 && colok) *reinterpret_cast<float4*>(const_cast<float*>(piece_ptr(a, c, q0)) + 4 * lane) =
        make_float4(g[0], g[1], g[2], g[3]);
    __threadfence();
    group_sync(0, T);
    if (tid == 0) *s_flag = atomicAdd(a.long_done + item, 1) == nseg - 1;
    group_sync(0, T);
    if (!*s_flag) return;
    __threadfence();
    if (tid < 32) {
        float gs[4] = {0.f, 0.f, 0.f, 0.f}, gc[4] = {0.f, 0.f, 0.f, 0.f};
        if (colok) {
            for (int sg = 0; sg < nseg; ++sg) {
                const float4 v = __ldcg(reinterpret_cast<const float4*>(piece_ptr(a, c, (int64_t)sg * P / nseg) + 4 * lane));
                kahan_add(gs[0], gc[0], v.x);
                kahan_add(gs[1], gc[1], v.y);
                kahan_add(gs[2], gc[2], v.z);
                kahan_add(gs[3], gc[3], v.w);
            }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) g[q] = __fsub_rn(gs[q], gc[q]);
        apply_row(a, tb, key, g, lane, colok);
        if (lane == 0) a.long_done[item] = 0;   // ready for the next backward
    }
}

// Persistent blocks of kCombineThreads over the runs registered as split,
// taking work from counters (split_count[2] for long rows, [3] for short
// ones): a block first adds long rows with all its warps, then works as
// kCombineGroups independent groups (named barriers 1..) on short rows.
__global__ void __launch_bounds__(kCombineThreads) reduce_update_combine(ReduceArgs a)
{
    __shared__ int64_t s_last[kCombineGroups];
    __shared__ int s_item[kCombineGroups];
    __shared__ int s_flag;
    __shared__ float part[kCombineThreads / 32][kMaxDim];
    const int nlong = a.split_count[1], nshort = a.split_count[0];
    for (;;) {
        if (threadIdx.x == 0) s_item[0] = atomicAdd(a.split_count + 2, 1);
        group_sync(0, kCombineThreads);
        const int task = s_item[0];
        if (task >= nlong * kLongSegs) break;
        combine_long_segment(a, task / kLongSegs, task % kLongSegs, part, &s_flag);
        group_sync(0, kCombineThreads);
    }
    constexpr int kGT = kCombineThreads / kCombineGroups;
    const int g = threadIdx.x / kGT, tid = threadIdx.x % kGT;
    group_sync(0, kCombineThreads);   // every thread has read s_item[0]
    for (;;) {
        if (tid == 0) s_item[g] = atomicAdd(a.split_count + 3, 1);
        group_sync(1 + g, kGT);
        const int item = s_item[g];
        if (item >= nshort) break;
        combine_run(a, (int64_t)a.split_list[item] + 1, s_last[g], part, 1 + g, kGT, tid, g * (kGT / 32));
        group_sync(1 + g, kGT);
    }
}
}  // namespace

int launch_reduce_update(const ReduceArgs& a, cudaStream_t st)
{
    if (a.n <= 0 || a.nchunks <= 0) return 0;
    if (cudaMemsetAsync(a.split_count, 0, 4 * sizeof(int), st) != cudaSuccess) return -1;
    const int64_t threads = a.nchunks * 32;
    const unsigned blocks = (unsigned)((threads + kThreads - 1) / kThreads);
    const size_t smem = sizeof(uint32_t) * (size_t)(kThreads / 32) * (size_t)warp_words(a.chunk);
    ChunkKernel kernel = nullptr;
    if (a.uni_dtype == EMB_F32) kernel = chunks_kernel_f32(a);
    else if (a.uni_dtype == EMB_F16) kernel = chunks_kernel_f16(a);
    else if (a.uni_dtype == EMB_BF16) kernel = chunks_kernel_bf16(a);
    if (!kernel) kernel = chunks_kernel<AnyLayer>(a);
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return -1;
    kernel<<<blocks, kThreads, smem, st>>>(a);
    int launched = 1;
    if (a.nchunks > 1) {
        int dev = 0, sms = 152;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        const int64_t cap = (int64_t)kCombineBlocksPerSM * sms;
        const int64_t grid = (a.nchunks - 1) < cap ? (a.nchunks - 1) : cap;
        reduce_update_combine<<<(unsigned)grid, kCombineThreads, 0, st>>>(a);
        ++launched;
    }
    if (cudaGetLastError() != cudaSuccess) return -1;
    return launched;
}

}  // namespace emb
