// k_reduce instantiations for fp32 replicas.
#define launch_reduce_dtype launch_reduce_f32
#define launch_reduce_acc_dtype launch_reduce_acc_f32
#define launch_accumulate_dtype launch_accumulate_f32
#define GAR_DTYPE F32
#include "gar_reduce.inc"
