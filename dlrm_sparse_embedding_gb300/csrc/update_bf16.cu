// Chunk kernels of the reduction for layers whose tables all store bf16 rows (master copies read per table)
// and share one optimizer and one pooling.
#include "reduce_chunks.cuh"

namespace emb {

ChunkKernel chunks_kernel_bf16(const ReduceArgs& a)
{
    if (a.uni_dtype != EMB_BF16) return nullptr;
    return chunks_kernel_uniform<EMB_BF16, -1>(a);
}

}  // namespace emb
