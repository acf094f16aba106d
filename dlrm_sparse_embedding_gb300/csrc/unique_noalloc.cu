// emb_unique_noalloc: the stand-alone unique for callers that cannot allocate
// device memory when they call it.
//
// Its scratch is one file-scope device array of fixed size, so the call itself
// performs no allocation of any kind.  Every GPU that loads this library holds
// the array (kNoAllocScratchBytes) until the process exits.  The array's
// device address is looked up once per device (cudaGetSymbolAddress, with that
// device current) on the first call made on that device.  The computation is
// exactly emb_unique's, run on that array instead of a caller workspace.
#include <mutex>

#include "emb_internal.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(12) << 20;  // fits emb_unique's workspace for the maximum n
constexpr int kMaxDevices = 64;

// The scratch.  Host code must not use this name as an address: on the host it
// is only a stand-in for the symbol, so it is passed to cudaGetSymbolAddress
// and never to a kernel.
static __device__ __align__(256) unsigned char g_unique_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up on first use.
int scratch_for_current_device(void** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return EMB_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return EMB_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_unique_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return EMB_ERR_CUDA;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return EMB_OK;
}

}  // namespace

namespace emb {
bool unique_args_valid(const int64_t* keys, int64_t n, const int64_t* unique, const int32_t* inverse,
                       const int32_t* counts, const int32_t* seg_offsets, const int64_t* num_unique);   // layer.cu
}

extern "C" int emb_unique_noalloc(const int64_t* keys, int64_t n, int64_t* unique, int32_t* inverse,
                                  int32_t* counts, int32_t* seg_offsets, int64_t* num_unique, void* stream)
{
    if (n > EMB_UNIQUE_NOALLOC_MAX_KEYS || !emb::unique_args_valid(keys, n, unique, inverse, counts, seg_offsets, num_unique))
        return EMB_ERR_INVALID_ARG;
    size_t need = 0;
    if (emb_unique_workspace(n, &need) != EMB_OK || need > kNoAllocScratchBytes) return EMB_ERR_INVALID_ARG;
    void* scratch = nullptr;
    const int rc = scratch_for_current_device(&scratch);
    if (rc != EMB_OK) return rc;
    // Nothing in the scratch has to start at zero: every buffer emb_unique uses
    // is fully written before it is read within the call.
    return emb_unique(keys, n, unique, inverse, counts, seg_offsets, num_unique, scratch, kNoAllocScratchBytes,
                      stream);
}
