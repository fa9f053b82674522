// k_reduce instantiations (no SGD step) for bf16 replicas.
#define GAR_LAUNCH launch_reduce_plain_bf16
#define GAR_DTYPE BF16
#define GAR_PART 0
#include "gar_reduce.inc"
