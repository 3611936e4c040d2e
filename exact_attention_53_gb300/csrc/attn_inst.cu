// One (head_dim, dtype, causal) instantiation of the attention forward kernel
// per object file, selected by -DATTN_D=<64|128|256> -DATTN_BF16=<0|1>
// -DATTN_CAUSAL=<0|1> [-DATTN_SPLIT=1, full attention only], so the
// instantiations compile in parallel.
#include "attn_fwd.cuh"

#if !defined(ATTN_D) || !defined(ATTN_BF16) || !defined(ATTN_CAUSAL)
#error "compile with -DATTN_D, -DATTN_BF16 and -DATTN_CAUSAL"
#endif
#ifndef ATTN_SPLIT
#define ATTN_SPLIT 0
#endif

namespace attn {
template cudaError_t launch_attn_fwd<ATTN_D, (ATTN_BF16 != 0), (ATTN_CAUSAL != 0), (ATTN_SPLIT != 0)>(
    const FwdArgs&, cudaStream_t);
}
