// k_reduce instantiations for bf16 replicas.
#define launch_reduce_dtype launch_reduce_bf16
#define GAR_DTYPE BF16
#include "gar_reduce.inc"
