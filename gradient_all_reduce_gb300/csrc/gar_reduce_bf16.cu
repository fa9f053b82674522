// k_reduce instantiations for bf16 replicas.
#define launch_reduce_dtype launch_reduce_bf16
#define launch_reduce_acc_dtype launch_reduce_acc_bf16
#define launch_accumulate_dtype launch_accumulate_bf16
#define GAR_DTYPE BF16
#include "gar_reduce.inc"
