// Chunk kernels of the reduction for layers whose tables all store fp16 rows (master copies read per table)
// and share one optimizer and one pooling.
#include "reduce_chunks.cuh"

namespace emb {

ChunkKernel chunks_kernel_f16(const ReduceArgs& a)
{
    if (a.uni_dtype != EMB_F16) return nullptr;
    return chunks_kernel_uniform<EMB_F16, -1>(a);
}

}  // namespace emb
