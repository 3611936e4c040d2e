// One (head_dim, dtype, causal) instantiation of the attention backward per
// object file, selected by -DATTN_D=<64|128|256> -DATTN_BF16=<0|1>
// -DATTN_CAUSAL=<0|1>, so the instantiations compile in parallel.
#include "attn_bwd.cuh"

#if !defined(ATTN_D) || !defined(ATTN_BF16) || !defined(ATTN_CAUSAL)
#error "compile with -DATTN_D, -DATTN_BF16 and -DATTN_CAUSAL"
#endif

namespace attn {
template cudaError_t launch_attn_bwd<ATTN_D, (ATTN_BF16 != 0), (ATTN_CAUSAL != 0)>(const BwdArgs&,
                                                                                    cudaStream_t);
}
