// moe_layer_tk1.cu -- the layer kernel instantiations of top-k class 1 (one
// translation unit per class, so the four compile in parallel).
#include "moe_layer_kernel.cuh"

namespace moe {
void *layer_kernel_tk1(int mc_gu, int mc_d) { return layer_kernel_table<1>(mc_gu, mc_d); }
}  // namespace moe
