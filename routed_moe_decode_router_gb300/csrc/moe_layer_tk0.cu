// moe_layer_tk0.cu -- the layer kernel instantiations of top-k class 0 with the
// tensor-core expert projections (one translation unit per class and
// variant, so the eight compile in parallel).
#include "moe_layer_kernel.cuh"

namespace moe {
void *layer_kernel_tk0(int mc_gu, int mc_d) { return layer_kernel_table<0, false>(mc_gu, mc_d); }
size_t layer_fixed_smem_bytes() { return kLayerSmemFixed; }
}  // namespace moe
