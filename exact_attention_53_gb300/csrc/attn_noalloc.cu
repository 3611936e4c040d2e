// Built-in scratch for attn_fwd_splitkv_noalloc.
//
// A fixed device array in its own translation unit: under CUDA's lazy module
// loading (the default) its memory is reserved only in processes that call the
// allocation-free entry point.  The host looks its address up with
// cudaGetSymbolAddress from this file, where the symbol is visible.
#pragma GCC visibility push(default)    // the C ABI is the library's only export
#include "attn.h"
#pragma GCC visibility pop
#include "attn_launch.h"

static __device__ __align__(256) unsigned char g_splitkv_scratch[ATTN_NOALLOC_SCRATCH_BYTES];

namespace attn {

cudaError_t noalloc_scratch_address(void** ptr) {
    return cudaGetSymbolAddress(ptr, g_splitkv_scratch);
}

}  // namespace attn
