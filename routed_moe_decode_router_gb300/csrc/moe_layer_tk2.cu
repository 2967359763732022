// moe_layer_tk2.cu -- the layer kernel instantiations of top-k class 2 with the
// tensor-core expert projections (one translation unit per class and
// variant, so the eight compile in parallel).
#include "moe_layer_kernel.cuh"

namespace moe {
void *layer_kernel_tk2(int mc_gu, int mc_d) { return layer_kernel_table<2, false>(mc_gu, mc_d); }
}  // namespace moe
