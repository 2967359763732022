// moe_layer_tk1_t.cu -- the layer kernel instantiations of top-k class 1
// for down projections in the t layout (the fused one-row form, both
// projection variants), in a translation unit of their own so that they
// compile in parallel with the others.
#include "moe_layer_kernel.cuh"

namespace moe {
void *layer_kernel_tk1_t(int mc_gu, bool gv) { return layer_kernel_t_table<1>(mc_gu, gv); }
}  // namespace moe
