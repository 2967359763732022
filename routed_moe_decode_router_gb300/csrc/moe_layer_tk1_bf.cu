// moe_layer_tk1_bf.cu -- the layer kernel instantiations of top-k class 1
// for BF16 expert matrices (tensor-core projections), in a translation unit
// of their own so that they compile in parallel with the others.
#include "moe_layer_kernel.cuh"

namespace moe {
void *layer_kernel_tk1_bf(int mc_gu, int mc_d) { return layer_kernel_table<1, false, 2>(mc_gu, mc_d); }
}  // namespace moe
