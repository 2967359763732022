// moe_layer_tk1.cu -- the layer kernel instantiations of top-k class 1 with the
// tensor-core expert projections (one translation unit per class and
// variant, so the eight compile in parallel).
#include "moe_layer_kernel.cuh"

namespace moe {
void *layer_kernel_tk1(int mc_gu, int mc_d) { return layer_kernel_table<1, false>(mc_gu, mc_d); }
}  // namespace moe
