// Instantiations of the gradient-reading kernels for fp16 gradients.
#define ZDP_GT ZDP_FP16
#define ZDP_GT_IS_BF16 0
#include "kernels_grad.inc"
