// Instantiations of the gradient-reading kernels for bf16 gradients.
#define ZDP_GT ZDP_BF16
#define ZDP_GT_IS_BF16 1
#include "kernels_grad.inc"
