// Chunk kernels of the reduction for layers whose tables all store fp32 rows (fp32 tables have no master copy)
// and share one optimizer and one pooling.
#include "reduce_chunks.cuh"

namespace emb {

ChunkKernel chunks_kernel_f32(const ReduceArgs& a)
{
    if (a.uni_dtype != EMB_F32) return nullptr;
    return chunks_kernel_uniform<EMB_F32, 0>(a);
}

}  // namespace emb
