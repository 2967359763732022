// moe_layer_tk3_kp.cu -- the layer kernel instantiations of top-k class 3
// for FP8 and BF16 expert matrices whose down tiles come in K-parts, in a
// translation unit of their own (a module apart from the instantiations that
// never need K-parts).
#include "moe_layer_kernel.cuh"

namespace moe {
void *layer_kernel_tk3_kp(int fmt, int mc_gu, int mc_d) {
    return fmt == MOE_EXPERT_FP8 ? layer_kernel_kp_table<3, MOE_EXPERT_FP8>(mc_gu, mc_d)
                                 : layer_kernel_kp_table<3, MOE_EXPERT_BF16>(mc_gu, mc_d);
}
}  // namespace moe
