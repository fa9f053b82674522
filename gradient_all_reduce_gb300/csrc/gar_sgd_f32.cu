// k_reduce instantiations with the fused SGD step for fp32 replicas.
#define GAR_LAUNCH launch_reduce_sgd_f32
#define GAR_DTYPE F32
#define GAR_PART 1
#include "gar_reduce.inc"
