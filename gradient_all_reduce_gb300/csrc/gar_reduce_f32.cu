// k_reduce instantiations (no SGD step) for fp32 replicas.
#define GAR_LAUNCH launch_reduce_plain_f32
#define GAR_DTYPE F32
#define GAR_PART 0
#include "gar_reduce.inc"
