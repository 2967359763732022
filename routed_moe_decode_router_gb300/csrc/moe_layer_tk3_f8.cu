// moe_layer_tk3_f8.cu -- the layer kernel instantiations of top-k class 3
// for FP8 expert matrices (tensor-core projections), in a translation unit
// of their own so that they compile in parallel with the others.
#include "moe_layer_kernel.cuh"

namespace moe {
void *layer_kernel_tk3_f8(int mc_gu, int mc_d) { return layer_kernel_table<3, false, 1>(mc_gu, mc_d); }
}  // namespace moe
