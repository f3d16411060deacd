// The single-pass checked step for fp16 gradients.
#define ZDP_GT ZDP_FP16
#define ZDP_GT_IS_BF16 0
#include "zdp_coop.inc"
