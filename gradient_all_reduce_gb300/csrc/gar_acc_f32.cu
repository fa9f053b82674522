// Accumulation kernel instantiations (no_sync) for fp32 gradients.
#define GAR_LAUNCH_ACC launch_reduce_acc_f32
#define GAR_LAUNCH_ACCUMULATE launch_accumulate_f32
#define GAR_DTYPE F32
#define GAR_PART 2
#include "gar_reduce.inc"
