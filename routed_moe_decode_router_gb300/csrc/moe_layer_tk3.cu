// moe_layer_tk3.cu -- the layer kernel instantiations of top-k class 3 (one
// translation unit per class, so the four compile in parallel).
#include "moe_layer_kernel.cuh"

namespace moe {
void *layer_kernel_tk3(int mc_gu, int mc_d) { return layer_kernel_table<3>(mc_gu, mc_d); }
}  // namespace moe
