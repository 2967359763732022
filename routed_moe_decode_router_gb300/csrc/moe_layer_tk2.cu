// moe_layer_tk2.cu -- the layer kernel instantiations of top-k class 2 (one
// translation unit per class, so the four compile in parallel).
#include "moe_layer_kernel.cuh"

namespace moe {
void *layer_kernel_tk2(int mc_gu, int mc_d) { return layer_kernel_table<2>(mc_gu, mc_d); }
}  // namespace moe
