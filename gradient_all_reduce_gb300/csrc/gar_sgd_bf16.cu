// k_reduce instantiations with the fused SGD step for bf16 replicas.
#define GAR_LAUNCH launch_reduce_sgd_bf16
#define GAR_DTYPE BF16
#define GAR_PART 1
#include "gar_reduce.inc"
