// Accumulation kernel instantiations (no_sync) for bf16 gradients.
#define GAR_LAUNCH_ACC launch_reduce_acc_bf16
#define GAR_LAUNCH_ACCUMULATE launch_accumulate_bf16
#define GAR_DTYPE BF16
#define GAR_PART 2
#include "gar_reduce.inc"
