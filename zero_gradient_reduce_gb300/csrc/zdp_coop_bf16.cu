// The single-pass checked step for bf16 gradients.
#define ZDP_GT ZDP_BF16
#define ZDP_GT_IS_BF16 1
#include "zdp_coop.inc"
