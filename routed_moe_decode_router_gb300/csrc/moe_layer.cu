// moe_layer.cu -- host side of the layer kernel: shared-memory sizing,
// kernel selection (MC_GU, MC_D, top-k class, projection variant) and the
// cooperative, PDL launch.  The kernel itself is in moe_layer_kernel.cuh,
// instantiated in moe_layer_tk0.cu .. moe_layer_tk3.cu (tensor-core
// projections), moe_layer_tk0_gv.cu .. moe_layer_tk3_gv.cu (the one-row
// CUDA-core GEMV), moe_layer_tk0_t.cu .. moe_layer_tk3_t.cu (the fused
// one-row form for down projections in the t layout, both variants) and
// moe_layer_tk*_f8.cu / moe_layer_tk*_bf.cu (FP8 and BF16 expert matrices)
// and moe_layer_tk*_kp.cu (FP8 / BF16 with down tiles in K-parts).
#include <cuda_runtime.h>

#include "moe_layout.h"

namespace moe {

void *layer_kernel_tk0(int mc_gu, int mc_d);
void *layer_kernel_tk1(int mc_gu, int mc_d);
void *layer_kernel_tk2(int mc_gu, int mc_d);
void *layer_kernel_tk3(int mc_gu, int mc_d);
void *layer_kernel_tk0_gv(int mc_gu, int mc_d);
void *layer_kernel_tk1_gv(int mc_gu, int mc_d);
void *layer_kernel_tk2_gv(int mc_gu, int mc_d);
void *layer_kernel_tk3_gv(int mc_gu, int mc_d);
void *layer_kernel_tk0_f8(int mc_gu, int mc_d);
void *layer_kernel_tk1_f8(int mc_gu, int mc_d);
void *layer_kernel_tk2_f8(int mc_gu, int mc_d);
void *layer_kernel_tk3_f8(int mc_gu, int mc_d);
void *layer_kernel_tk0_bf(int mc_gu, int mc_d);
void *layer_kernel_tk1_bf(int mc_gu, int mc_d);
void *layer_kernel_tk2_bf(int mc_gu, int mc_d);
void *layer_kernel_tk3_bf(int mc_gu, int mc_d);
void *layer_kernel_tk0_t(int mc_gu, bool gv);
void *layer_kernel_tk1_t(int mc_gu, bool gv);
void *layer_kernel_tk2_t(int mc_gu, bool gv);
void *layer_kernel_tk3_t(int mc_gu, bool gv);
void *layer_kernel_tk0_kp(int fmt, int mc_gu, int mc_d);
void *layer_kernel_tk1_kp(int fmt, int mc_gu, int mc_d);
void *layer_kernel_tk2_kp(int fmt, int mc_gu, int mc_d);
void *layer_kernel_tk3_kp(int fmt, int mc_gu, int mc_d);
size_t layer_fixed_smem_bytes();

size_t layer_smem_bytes(int stages, uint32_t slot_bytes) {
    return layer_fixed_smem_bytes() + (size_t)stages * slot_bytes + 2 * sizeof(uint64_t) * stages;
}

// Top-k class of a router width (the top-k keeps E / 32 candidates per lane
// in registers: 4, 8, 16 or two lists of 16).
static int topk_class(int E) { return E <= 128 ? 0 : (E <= 256 ? 1 : (E <= 512 ? 2 : 3)); }

static void *layer_kernel(int mc_gu, int mc_d, int tk, bool gv, bool tl, int fmt,
                          bool kp = false) {
    if (kp) {
        switch (tk) {
        case 0: return layer_kernel_tk0_kp(fmt, mc_gu, mc_d);
        case 1: return layer_kernel_tk1_kp(fmt, mc_gu, mc_d);
        case 2: return layer_kernel_tk2_kp(fmt, mc_gu, mc_d);
        default: return layer_kernel_tk3_kp(fmt, mc_gu, mc_d);
        }
    }
    if (fmt == MOE_EXPERT_FP8) {
        switch (tk) {
        case 0: return layer_kernel_tk0_f8(mc_gu, mc_d);
        case 1: return layer_kernel_tk1_f8(mc_gu, mc_d);
        case 2: return layer_kernel_tk2_f8(mc_gu, mc_d);
        default: return layer_kernel_tk3_f8(mc_gu, mc_d);
        }
    }
    if (fmt == MOE_EXPERT_BF16) {
        switch (tk) {
        case 0: return layer_kernel_tk0_bf(mc_gu, mc_d);
        case 1: return layer_kernel_tk1_bf(mc_gu, mc_d);
        case 2: return layer_kernel_tk2_bf(mc_gu, mc_d);
        default: return layer_kernel_tk3_bf(mc_gu, mc_d);
        }
    }
    if (tl) {
        switch (tk) {
        case 0: return layer_kernel_tk0_t(mc_gu, gv);
        case 1: return layer_kernel_tk1_t(mc_gu, gv);
        case 2: return layer_kernel_tk2_t(mc_gu, gv);
        default: return layer_kernel_tk3_t(mc_gu, gv);
        }
    }
    switch (tk) {
    case 0: return gv ? layer_kernel_tk0_gv(mc_gu, mc_d) : layer_kernel_tk0(mc_gu, mc_d);
    case 1: return gv ? layer_kernel_tk1_gv(mc_gu, mc_d) : layer_kernel_tk1(mc_gu, mc_d);
    case 2: return gv ? layer_kernel_tk2_gv(mc_gu, mc_d) : layer_kernel_tk2(mc_gu, mc_d);
    default: return gv ? layer_kernel_tk3_gv(mc_gu, mc_d) : layer_kernel_tk3(mc_gu, mc_d);
    }
}

cudaError_t set_layer_smem_limit(int bytes) {
    for (int v = 0; v < 2; ++v)
        for (int t = 0; t < 4; ++t)
            for (int a = 1; a <= 4; ++a)
                for (int b = 1; b <= 4; ++b)
                    // (MC_D = 1 also stands for the t-layout form of this MC_GU)
                    for (int tl = 0; tl < (b == 1 ? 2 : 1); ++tl) {
                        cudaError_t e = cudaFuncSetAttribute(
                            layer_kernel(a, b, t, v != 0, tl != 0, MOE_EXPERT_NVFP4),
                            cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
                        if (e != cudaSuccess) return e;
                    }
    // FP8 and BF16 experts: tensor-core projections, output-major down
    for (int f = MOE_EXPERT_FP8; f <= MOE_EXPERT_BF16; ++f)
        for (int t = 0; t < 4; ++t)
            for (int a = 1; a <= 4; ++a)
                for (int b = 1; b <= 4; ++b) {
                    cudaError_t e = cudaFuncSetAttribute(layer_kernel(a, b, t, false, false, f),
                                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                         bytes);
                    if (e != cudaSuccess) return e;
                    void *kp = layer_kernel(a, b, t, false, false, f, true);
                    if (kp) {
                        e = cudaFuncSetAttribute(kp, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
                        if (e != cudaSuccess) return e;
                    }
                }
    return cudaSuccess;
}

cudaError_t launch_layer(const LayerParams &p, int grid, size_t smem, int mc_gu, int mc_d,
                         bool gemv, bool t_layout, int expert_fmt, cudaStream_t stream) {
    // FP8 / BF16 down tiles in K-parts (down_pc below the widest
    // intermediate's chunk count) take the K-part instantiations
    const int inter_max = p.has_shared && p.Is > p.I ? p.Is : p.I;
    const bool kp = !t_layout && expert_fmt != MOE_EXPERT_NVFP4 && p.down_pc < inter_max / kChunk;
    void *fn = layer_kernel(mc_gu, mc_d, topk_class(p.E), gemv, t_layout, expert_fmt, kp);
    if (!fn) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kLayerBlockThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    void *args[] = {const_cast<LayerParams *>(&p)};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace moe
