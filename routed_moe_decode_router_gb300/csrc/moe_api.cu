// moe_api.cu -- host side of the C ABI declared in include/moe_router.h:
// argument checks (all before the first launch), workspace layout, the launch
// of the persistent layer kernel (programmatic dependent launch on the
// caller's stream) and of the stage kernels behind moe_route / moe_union.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "moe_layout.h"

namespace moe {
cudaError_t launch_route(const RouteParams &p, cudaStream_t stream);
cudaError_t launch_union(const UnionParams &p, cudaStream_t stream);
cudaError_t launch_layer(const LayerParams &p, int grid, size_t smem, int mc_gu, int mc_d,
                         bool gemv, bool t_layout, int expert_fmt, cudaStream_t stream);
cudaError_t launch_t_layout(const uint8_t *packed, const uint8_t *scales, int count, int n_out,
                            int k_in, uint8_t *packed_t, uint8_t *scales_t, cudaStream_t stream);
cudaError_t set_layer_smem_limit(int bytes);
size_t layer_smem_bytes(int stages, uint32_t slot_bytes);
}  // namespace moe

using namespace moe;

namespace {

thread_local char g_err[512];

moe_status fail(moe_status s, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return s;
}

moe_status ok() {
    g_err[0] = 0;
    return MOE_OK;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Per-device facts, looked up once.
struct DevInfo {
    int sms = 0;
    int smem_optin = 0;
    bool attrs_set = false;
};
std::mutex g_mu;
DevInfo g_dev[64];

moe_status device_info(DevInfo **out) {
    int d = 0;
    cudaError_t e = cudaGetDevice(&d);
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (d < 0 || d >= 64) return fail(MOE_ERR_CUDA, "device ordinal %d out of range", d);
    std::lock_guard<std::mutex> lk(g_mu);
    DevInfo &di = g_dev[d];
    if (!di.attrs_set) {
        if ((e = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, d)) !=
                cudaSuccess ||
            (e = cudaDeviceGetAttribute(&di.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                        d)) != cudaSuccess)
            return fail(MOE_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
        if ((e = set_layer_smem_limit(di.smem_optin - 1024)) != cudaSuccess)
            return fail(MOE_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
        di.attrs_set = true;
    }
    *out = &di;
    return MOE_OK;
}

moe_status check_cfg(const moe_config *c) {
    if (!c) return fail(MOE_ERR_INVALID_ARG, "cfg is NULL");
    if (c->hidden < kChunk || c->hidden > MOE_MAX_HIDDEN || c->hidden % kChunk)
        return fail(MOE_ERR_INVALID_ARG, "hidden=%d: must be a multiple of %d in [%d, %d]",
                    c->hidden, kChunk, kChunk, MOE_MAX_HIDDEN);
    if (c->num_experts < 1 || c->num_experts > MOE_MAX_EXPERTS)
        return fail(MOE_ERR_INVALID_ARG, "num_experts=%d: must be in [1, %d]", c->num_experts,
                    MOE_MAX_EXPERTS);
    if (c->router_width != c->num_experts)
        return fail(MOE_ERR_UNSUPPORTED,
                    "router_width=%d differs from num_experts=%d: zero-computation experts "
                    "are not supported by this path",
                    c->router_width, c->num_experts);
    if (c->top_k < 1 || c->top_k > c->num_experts || c->top_k > MOE_CHUNK_IDS)
        return fail(MOE_ERR_INVALID_ARG, "top_k=%d: must be in [1, min(num_experts, %d)]",
                    c->top_k, MOE_CHUNK_IDS);
    if (c->moe_inter < kChunk || c->moe_inter % kChunk || c->moe_inter > 4 * kConsumerWarps * kChunk)
        return fail(MOE_ERR_INVALID_ARG, "moe_inter=%d: must be a multiple of %d in [%d, %d]",
                    c->moe_inter, kChunk, kChunk, 4 * kConsumerWarps * kChunk);
    if (c->has_shared != 0 && c->has_shared != 1)
        return fail(MOE_ERR_INVALID_ARG, "has_shared must be 0 or 1");
    if (c->has_shared &&
        (c->shared_inter < kChunk || c->shared_inter % kChunk ||
         c->shared_inter > 4 * kConsumerWarps * kChunk))
        return fail(MOE_ERR_INVALID_ARG, "shared_inter=%d: must be a multiple of %d in [%d, %d]",
                    c->shared_inter, kChunk, kChunk, 4 * kConsumerWarps * kChunk);
    if (c->scoring != MOE_SCORING_SOFTMAX && c->scoring != MOE_SCORING_SIGMOID)
        return fail(MOE_ERR_INVALID_ARG, "scoring=%d: must be softmax (0) or sigmoid (1)",
                    c->scoring);
    if (c->scoring == MOE_SCORING_SOFTMAX && c->routed_scaling_factor != 1.0f)
        return fail(MOE_ERR_UNSUPPORTED,
                    "routed_scaling_factor=%g with softmax scoring: the softmax top-k takes "
                    "no scaling factor (must be 1)",
                    (double)c->routed_scaling_factor);
    if (!std::isfinite(c->routed_scaling_factor))
        return fail(MOE_ERR_INVALID_ARG, "routed_scaling_factor is not finite");
    if (c->router_fmt != MOE_ROUTER_BF16 && c->router_fmt != MOE_ROUTER_NVFP4)
        return fail(MOE_ERR_INVALID_ARG, "router_fmt=%d: must be bf16 (0) or nvfp4 (1)",
                    c->router_fmt);
    if ((c->norm_topk_prob | c->shared_gate | c->per_row_mode | c->gemv_lever | c->t_layout) & ~1)
        return fail(MOE_ERR_INVALID_ARG,
                    "norm_topk_prob, shared_gate, per_row_mode, gemv_lever, t_layout are 0/1");
    if (c->expert_fmt != MOE_EXPERT_NVFP4 && c->expert_fmt != MOE_EXPERT_FP8 &&
        c->expert_fmt != MOE_EXPERT_BF16)
        return fail(MOE_ERR_INVALID_ARG, "expert_fmt=%d: must be nvfp4 (0), fp8 (1) or bf16 (2)",
                    c->expert_fmt);
    if (c->t_layout && c->expert_fmt != MOE_EXPERT_NVFP4)
        return fail(MOE_ERR_UNSUPPORTED, "the t layout holds NVFP4 down projections only");
    return MOE_OK;
}

moe_status check_rows(const moe_config *c, int rows) {
    if (rows < 1 || rows > MOE_MAX_ROWS)
        return fail(MOE_ERR_INVALID_ARG, "rows=%d: must be in [1, %d]", rows, MOE_MAX_ROWS);
    if (rows * c->top_k > MOE_MAX_IDS)
        return fail(MOE_ERR_UNSUPPORTED, "rows*top_k=%d exceeds %d ids (the union's capacity)",
                    rows * c->top_k, MOE_MAX_IDS);
    return MOE_OK;
}

// Rows of one sub-chunk: at most 8, and at most 64 ids (one union block).
int chunk_rows(const moe_config *c) {
    const int r = MOE_CHUNK_IDS / c->top_k;
    return r < MOE_CHUNK_ROWS ? r : MOE_CHUNK_ROWS;
}

UnionParams union_params(const moe_config *c, const moe_weights *w, const int32_t *ids, int rows,
                         const WsPtrs &wp, moe_union_table *out) {
    UnionParams p{};
    p.E = c->num_experts;
    p.k = c->top_k;
    p.rows = rows;
    p.per_row_mode = c->per_row_mode;
    p.has_tables = w != nullptr;
    p.has_shared = c->has_shared;
    p.has_scales = c->expert_fmt == MOE_EXPERT_NVFP4;
    p.ids = ids;
    if (w) {
        p.gate = w->gate;
        p.up = w->up;
        p.down = w->down;
        p.sh_gate = w->shared_gate_proj;
        p.sh_up = w->shared_up_proj;
        p.sh_down = w->shared_down_proj;
    }
    p.ws = wp;
    p.out = out;
    return p;
}

moe_status check_ws(const moe_config *c, const void *ws, size_t ws_bytes, WsLayout *L) {
    *L = WsLayout::make(*c);
    if (!ws) return fail(MOE_ERR_WORKSPACE, "workspace is NULL");
    if (!aligned(ws, 256)) return fail(MOE_ERR_WORKSPACE, "workspace is not 256-byte aligned");
    if (ws_bytes < L->total)
        return fail(MOE_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, L->total);
    return MOE_OK;
}

// has_scales = 0 (FP8 and BF16 experts): the scales pointers are not read
// and may be NULL.
moe_status check_mat(const moe_nvfp4 &m, const char *name, bool has_scales = true) {
    if (!m.packed || (has_scales && !m.scales))
        return fail(MOE_ERR_INVALID_ARG, "%s: NULL pointer", name);
    if (!aligned(m.packed, 16) || (has_scales && !aligned(m.scales, 16)))
        return fail(MOE_ERR_INVALID_ARG, "%s: packed/scales must be 16-byte aligned", name);
    return MOE_OK;
}

moe_status check_table(const moe_expert_table &t, const char *name, bool has_scales) {
    if (!t.packed || (has_scales && !t.scales) || !t.scale2)
        return fail(MOE_ERR_INVALID_ARG, "%s expert table: NULL array", name);
    if (!aligned(t.packed, 8) || (has_scales && !aligned(t.scales, 8)) || !aligned(t.scale2, 4))
        return fail(MOE_ERR_INVALID_ARG, "%s expert table: misaligned array", name);
    return MOE_OK;
}

moe_status check_weights(const moe_config *c, const moe_weights *w, bool experts) {
    moe_status s;
    if (!w) return fail(MOE_ERR_INVALID_ARG, "weights is NULL");
    if (c->router_fmt == MOE_ROUTER_BF16) {
        if (!w->router_bf16 || !aligned(w->router_bf16, 16))
            return fail(MOE_ERR_INVALID_ARG, "router_bf16: NULL or not 16-byte aligned");
    } else if ((s = check_mat(w->router_nvfp4, "router_nvfp4")) != MOE_OK) {
        return s;
    }
    if (c->scoring == MOE_SCORING_SIGMOID && (!w->correction_bias || !aligned(w->correction_bias, 4)))
        return fail(MOE_ERR_INVALID_ARG, "sigmoid scoring needs correction_bias");
    if (c->has_shared && c->shared_gate &&
        (!w->shared_expert_gate || !aligned(w->shared_expert_gate, 16)))
        return fail(MOE_ERR_INVALID_ARG, "shared_gate=1 needs a 16-byte aligned shared_expert_gate");
    if (!experts) return MOE_OK;
    const bool sc = c->expert_fmt == MOE_EXPERT_NVFP4;
    if ((s = check_table(w->gate, "gate", sc)) != MOE_OK) return s;
    if ((s = check_table(w->up, "up", sc)) != MOE_OK) return s;
    if ((s = check_table(w->down, "down", sc)) != MOE_OK) return s;
    if (c->has_shared) {
        if ((s = check_mat(w->shared_gate_proj, "shared_gate_proj", sc)) != MOE_OK) return s;
        if ((s = check_mat(w->shared_up_proj, "shared_up_proj", sc)) != MOE_OK) return s;
        if ((s = check_mat(w->shared_down_proj, "shared_down_proj", sc)) != MOE_OK) return s;
    }
    return MOE_OK;
}

moe_status check_io(const void *x, const void *out, int rows, int H) {
    if (!x || !aligned(x, 16)) return fail(MOE_ERR_INVALID_ARG, "x: NULL or not 16-byte aligned");
    if (out) {
        if (!aligned(out, 16)) return fail(MOE_ERR_INVALID_ARG, "out: not 16-byte aligned");
        const char *a = static_cast<const char *>(x), *b = static_cast<const char *>(out);
        const size_t n = (size_t)rows * H * 2;
        if (a < b + n && b < a + n) return fail(MOE_ERR_INVALID_ARG, "x and out overlap");
    }
    return MOE_OK;
}

RouteParams route_params(const moe_config *c, const moe_weights *w, const uint16_t *x, int rows,
                         const WsPtrs &wp) {
    RouteParams p{};
    p.H = c->hidden;
    p.E = c->num_experts;
    p.k = c->top_k;
    p.rows = rows;
    p.scoring = c->scoring;
    p.norm = c->norm_topk_prob;
    p.router_fmt = c->router_fmt;
    p.has_shared = c->has_shared;
    p.shared_gated = c->has_shared && c->shared_gate;
    p.per_row_mode = c->per_row_mode;
    p.rsf = c->routed_scaling_factor;
    p.x = x;
    p.router_bf16 = w->router_bf16;
    p.router_fp4 = w->router_nvfp4;
    p.bias = w->correction_bias;
    p.sh_vec = w->shared_expert_gate;
    p.gate = w->gate;
    p.up = w->up;
    p.down = w->down;
    p.sh_gate = w->shared_gate_proj;
    p.sh_up = w->shared_up_proj;
    p.sh_down = w->shared_down_proj;
    p.ws = wp;
    return p;
}

}  // namespace

namespace moe {
// Record a refusal or error for moe_last_error() from another translation
// unit of the library.
moe_status set_error(moe_status s, const char *msg) { return fail(s, "%s", msg); }

// Every host check of moe_forward except the workspace's: configuration,
// rows, weights, x and out.  moe_forward_static runs it before it clears its
// own workspace, so that a refused call enqueues nothing there either.
moe_status check_forward_args(const moe_config *cfg, const moe_weights *w, const uint16_t *x,
                              const uint16_t *out, int rows) {
    moe_status s;
    if ((s = check_cfg(cfg)) != MOE_OK || (s = check_rows(cfg, rows)) != MOE_OK ||
        (s = check_weights(cfg, w, true)) != MOE_OK)
        return s;
    if (!out) return fail(MOE_ERR_INVALID_ARG, "out is NULL");
    return check_io(x, out, rows, cfg->hidden);
}
}  // namespace moe

extern "C" {

int moe_abi_version(void) { return MOE_ABI_VERSION; }

const char *moe_last_error(void) { return g_err; }

moe_status moe_check_config(const moe_config *cfg) {
    moe_status s = check_cfg(cfg);
    return s == MOE_OK ? ok() : s;
}

size_t moe_workspace_size(const moe_config *cfg) {
    if (check_cfg(cfg) != MOE_OK) return 0;
    return WsLayout::make(*cfg).total;
}

moe_status moe_workspace_init(void *ws, size_t ws_bytes, void *stream) {
    if (!ws || !aligned(ws, 256) || ws_bytes < sizeof(WsHeader))
        return fail(MOE_ERR_WORKSPACE, "workspace NULL, misaligned or too small");
    cudaError_t e = cudaMemsetAsync(ws, 0, ws_bytes, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "cudaMemsetAsync: %s", cudaGetErrorString(e));
    return ok();
}

moe_status moe_route(const moe_config *cfg, const moe_weights *w, const uint16_t *x, int rows,
                     int32_t *ids, float *wts, float *logits, void *ws, size_t ws_bytes,
                     void *stream) {
    moe_status s;
    WsLayout L;
    if ((s = check_cfg(cfg)) != MOE_OK || (s = check_rows(cfg, rows)) != MOE_OK ||
        (s = check_weights(cfg, w, false)) != MOE_OK ||
        (s = check_io(x, nullptr, rows, cfg->hidden)) != MOE_OK ||
        (s = check_ws(cfg, ws, ws_bytes, &L)) != MOE_OK)
        return s;
    if ((ids && !aligned(ids, 4)) || (wts && !aligned(wts, 4)) || (logits && !aligned(logits, 4)))
        return fail(MOE_ERR_INVALID_ARG, "ids / wts / logits must be 4-byte aligned");
    // one launch per sub-chunk of at most 8 rows
    const int cr = chunk_rows(cfg), H = cfg->hidden, E = cfg->num_experts, k = cfg->top_k;
    for (int r0 = 0; r0 < rows; r0 += cr) {
        const int n = rows - r0 < cr ? rows - r0 : cr;
        RouteParams p = route_params(cfg, w, x + (size_t)r0 * H, n, ws_ptrs(ws, L));
        p.row_base = r0;
        p.ids_out = ids ? ids + (size_t)r0 * k : nullptr;
        p.wts_out = wts ? wts + (size_t)r0 * k : nullptr;
        p.logits_out = logits ? logits + (size_t)r0 * E : nullptr;
        cudaError_t e = launch_route(p, static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "route launch: %s", cudaGetErrorString(e));
    }
    return ok();
}

moe_status moe_union(const moe_config *cfg, const moe_weights *w, const int32_t *ids, int rows,
                     moe_union_table *out, void *ws, size_t ws_bytes, void *stream) {
    moe_status s;
    WsLayout L;
    if ((s = check_cfg(cfg)) != MOE_OK || (s = check_rows(cfg, rows)) != MOE_OK ||
        (s = check_ws(cfg, ws, ws_bytes, &L)) != MOE_OK)
        return s;
    if (!ids || !aligned(ids, 4)) return fail(MOE_ERR_INVALID_ARG, "ids: NULL or misaligned");
    if (out && !aligned(out, 4)) return fail(MOE_ERR_INVALID_ARG, "out: misaligned");
    if (w && (s = check_weights(cfg, w, true)) != MOE_OK) return s;
    const UnionParams p = union_params(cfg, w, ids, rows, ws_ptrs(ws, L), out);
    cudaError_t e = launch_union(p, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "union launch: %s", cudaGetErrorString(e));
    return ok();
}

}  // extern "C"

static moe_status forward_impl(const moe_config *cfg, const moe_weights *w,
                               const uint16_t *x, uint16_t *out, int rows, void *ws,
                               size_t ws_bytes, void *stream, void *const *ev) {
    moe_status s;
    WsLayout L;
    if ((s = moe::check_forward_args(cfg, w, x, out, rows)) != MOE_OK ||
        (s = check_ws(cfg, ws, ws_bytes, &L)) != MOE_OK)
        return s;
    DevInfo *di;
    if ((s = device_info(&di)) != MOE_OK) return s;

    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    LayerParams lp{};
    lp.H = cfg->hidden;
    lp.E = cfg->num_experts;
    lp.k = cfg->top_k;
    lp.rows = rows;
    lp.I = cfg->moe_inter;
    lp.Is = cfg->has_shared ? cfg->shared_inter : 0;
    lp.scoring = cfg->scoring;
    lp.norm = cfg->norm_topk_prob;
    lp.router_fmt = cfg->router_fmt;
    lp.has_shared = cfg->has_shared;
    lp.shared_gated = cfg->has_shared && cfg->shared_gate;
    lp.per_row_mode = cfg->per_row_mode;
    lp.rsf = cfg->routed_scaling_factor;
    lp.x = x;
    lp.out = out;
    lp.router_bf16 = w->router_bf16;
    lp.router_fp4 = w->router_nvfp4;
    lp.bias = w->correction_bias;
    lp.sh_vec = w->shared_expert_gate;
    lp.gate = w->gate;
    lp.up = w->up;
    lp.down = w->down;
    lp.sh_gate = w->shared_gate_proj;
    lp.sh_up = w->shared_up_proj;
    lp.sh_down = w->shared_down_proj;
    lp.ws = ws_ptrs(ws, L);

    // Down units of 64 output rows ("wide") when every entry's intermediate
    // is 2 or 4 chunks of 128: the eight compute warps then split a unit's
    // chunks and 16-row tiles between them, instead of leaving half of them
    // without a chunk, and the unit's tile is one copy of twice the size.
    auto narrow = [](int inter) { return inter == 2 * kChunk || inter == 4 * kChunk; };
    const bool wide = narrow(cfg->moe_inter) && (!cfg->has_shared || narrow(cfg->shared_inter));
    lp.down_rows = wide ? 2 * kOutTile : kOutTile;
    // Otherwise, when every entry's intermediate is 8, 12 or 16 chunks, each
    // compute warp takes one of a unit's two 16-row tiles at a quarter of its
    // chunks ("split" units): the same work for every warp and four partial
    // sums a tile for the epilogue.
    auto quarters = [](int inter) {
        const int n = inter / kChunk;
        return n % 4 == 0 && n >= 8 && n <= 16;
    };
    lp.down_split = !wide && quarters(cfg->moe_inter) &&
                    (!cfg->has_shared || quarters(cfg->shared_inter));
    // Ring slot = one 16-row gate or up tile (16 x H/2 packed + 16 x H/16
    // scale bytes) or one down tile (down_rows x I/2 + down_rows x I/16); a
    // gate+up unit takes two slots, a down unit one.
    // In the t layout a unit's third slot holds its 16 rows of the
    // transposed down matrix (16 x H/2 + H bytes: the size of a gate tile),
    // and there are no down units.
    const bool tl = cfg->t_layout != 0;
    // bytes of one row of K inputs in the expert format, block scales included
    auto row_bytes = [cfg](int K) -> size_t {
        return cfg->expert_fmt == MOE_EXPERT_FP8 ? (size_t)K
               : cfg->expert_fmt == MOE_EXPERT_BF16 ? 2 * (size_t)K
                                                    : (size_t)K / 2 + (size_t)K / 16;
    };
    size_t gu_slot = (size_t)kTileRows * row_bytes(cfg->hidden);
    size_t d_slot = tl ? 0 : (size_t)lp.down_rows * row_bytes(L.inter_max);
    const int budget = di->smem_optin - 1024;
    // BF16 gate/up tiles that do not fit two ring slots are taken in two
    // K-halves (each half a whole number of 128-input chunks)
    lp.gu_halves = 1;
    if (cfg->expert_fmt == MOE_EXPERT_BF16 && layer_smem_bytes(2, (uint32_t)gu_slot) > (size_t)budget &&
        (cfg->hidden / kChunk) % 2 == 0) {
        lp.gu_halves = 2;
        gu_slot /= 2;
    }
    // FP8 / BF16 down tiles that do not fit two ring slots are taken in
    // K-parts of down_pc chunks (down_rows row segments per slot), as many
    // chunks per part as leave room for four slots
    lp.down_pc = L.inter_max / kChunk;
    if (cfg->expert_fmt != MOE_EXPERT_NVFP4 && !tl &&
        layer_smem_bytes(2, (uint32_t)gu_slot) <= (size_t)budget &&
        layer_smem_bytes(2, (uint32_t)d_slot) > (size_t)budget) {
        const size_t per_chunk = (size_t)lp.down_rows * row_bytes(kChunk);
        int pc = lp.down_pc;
        while (pc > 1 && layer_smem_bytes(4, (uint32_t)(gu_slot > per_chunk * pc ? gu_slot
                                                                          : per_chunk * pc)) >
                             (size_t)budget)
            --pc;
        if (wide) return fail(MOE_ERR_UNSUPPORTED, "wide down units do not fit the ring");
        lp.down_pc = pc;
        d_slot = per_chunk * pc;
    }
    lp.slot_bytes = (uint32_t)(gu_slot > d_slot ? gu_slot : d_slot);
    int S = 16;
    while (S > 2 && layer_smem_bytes(S, lp.slot_bytes) > (size_t)budget) --S;
    if (layer_smem_bytes(S, lp.slot_bytes) > (size_t)budget || (tl && S < 4))
        return fail(MOE_ERR_UNSUPPORTED, "stage ring does not fit in shared memory");
    if (tl && (di->sms > kMaxTCtas || cfg->hidden > 256 * di->sms))
        return fail(MOE_ERR_UNSUPPORTED,
                    "t layout: %d SMs (the workspace holds the partials of at most %d, and "
                    "each SM sums at most 256 outputs)", di->sms, kMaxTCtas);
    lp.stages = S;
    const int mc_gu = (cfg->hidden / kChunk + kConsumerWarps - 1) / kConsumerWarps;
    const int mc_d = lp.down_split ? L.inter_max / kChunk / 4
                                   : (L.inter_max / kChunk + kConsumerWarps - 1) / kConsumerWarps;
    if (lp.down_pc < L.inter_max / kChunk && !down_parts_possible(cfg->expert_fmt, mc_d))
        return fail(MOE_ERR_UNSUPPORTED, "down tiles in K-parts need more chunks per warp");

    // one launch per sub-chunk of at most 8 rows (64 ids), in row order; a
    // call of several sub-chunks then resolves the union of all its rows
    const int cr = tl ? 1 : chunk_rows(cfg), H = cfg->hidden;
    const int nchunks = (rows + cr - 1) / cr;
    cudaError_t e = cudaSuccess;
    if (ev) e = cudaEventRecord(static_cast<cudaEvent_t>(ev[0]), st);
    for (int c = 0; c < nchunks && e == cudaSuccess; ++c) {
        const int r0 = c * cr, n = rows - r0 < cr ? rows - r0 : cr;
        lp.rows = n;
        lp.row_base = r0;
        lp.publish_union = nchunks == 1;
        lp.x = x + (size_t)r0 * H;
        lp.out = out + (size_t)r0 * H;
        // gemv_lever applies per sub-chunk, so that a one-row last sub-chunk
        // gives the bytes of a one-row call
        e = launch_layer(lp, di->sms, layer_smem_bytes(S, lp.slot_bytes), mc_gu, tl ? 1 : mc_d,
                         n == 1 && cfg->gemv_lever && cfg->expert_fmt == MOE_EXPERT_NVFP4, tl,
                         cfg->expert_fmt, st);
    }
    if (e == cudaSuccess && nchunks > 1)
        e = launch_union(union_params(cfg, w, lp.ws.ids, rows, lp.ws, nullptr), st);
    if (e == cudaSuccess && ev) e = cudaEventRecord(static_cast<cudaEvent_t>(ev[1]), st);
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "layer launch: %s", cudaGetErrorString(e));
    return ok();
}

extern "C" {

moe_status moe_forward(const moe_config *cfg, const moe_weights *w, const uint16_t *x,
                       uint16_t *out, int rows, void *ws, size_t ws_bytes, void *stream) {
    return forward_impl(cfg, w, x, out, rows, ws, ws_bytes, stream, nullptr);
}

moe_status moe_nvfp4_to_t_layout(const uint8_t *packed, const uint8_t *scales, int count,
                                 int n_out, int k_in, uint8_t *packed_t, uint8_t *scales_t,
                                 void *stream) {
    if (count < 1) return fail(MOE_ERR_INVALID_ARG, "count=%d: must be at least 1", count);
    if (n_out < 16 || n_out > 65536 || n_out % 16 || k_in < 16 || k_in > 65536 || k_in % 16)
        return fail(MOE_ERR_INVALID_ARG,
                    "n_out=%d, k_in=%d: each must be a multiple of 16 in [16, 65536]", n_out, k_in);
    if (!packed || !scales || !packed_t || !scales_t)
        return fail(MOE_ERR_INVALID_ARG, "a matrix pointer is NULL");
    if (!aligned(packed, 16) || !aligned(scales, 16) || !aligned(packed_t, 16) ||
        !aligned(scales_t, 16))
        return fail(MOE_ERR_INVALID_ARG, "matrix pointers must be 16-byte aligned");
    const size_t pk = (size_t)count * n_out * (k_in / 2), sc = (size_t)count * n_out * (k_in / 16);
    auto overlap = [](const void *a, size_t na, const void *b, size_t nb) {
        const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
        return x < y + nb && y < x + na;
    };
    if (overlap(packed_t, pk, packed, pk) || overlap(packed_t, pk, scales, sc) ||
        overlap(scales_t, sc, packed, pk) || overlap(scales_t, sc, scales, sc) ||
        overlap(packed_t, pk, scales_t, sc))
        return fail(MOE_ERR_INVALID_ARG, "the t-layout outputs overlap each other or the inputs");
    const cudaError_t e = launch_t_layout(packed, scales, count, n_out, k_in, packed_t, scales_t,
                                          static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "t-layout launch: %s", cudaGetErrorString(e));
    return ok();
}

moe_status moe_forward_timed(const moe_config *cfg, const moe_weights *w, const uint16_t *x,
                             uint16_t *out, int rows, void *ws, size_t ws_bytes, void *stream,
                             void *const ev[2]) {
    if (!ev || !ev[0] || !ev[1]) return fail(MOE_ERR_INVALID_ARG, "two events are required");
    return forward_impl(cfg, w, x, out, rows, ws, ws_bytes, stream, ev);
}

moe_status moe_read_routing(const moe_config *cfg, const void *ws, size_t ws_bytes, int rows,
                            int32_t *ids, float *wts, moe_union_table *uni, void *stream) {
    moe_status s;
    WsLayout L;
    if ((s = check_cfg(cfg)) != MOE_OK || (s = check_rows(cfg, rows)) != MOE_OK ||
        (s = check_ws(cfg, ws, ws_bytes, &L)) != MOE_OK)
        return s;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const char *b = static_cast<const char *>(ws);
    const size_t n = (size_t)rows * cfg->top_k;
    cudaError_t e = cudaSuccess;
    if (ids && e == cudaSuccess)
        e = cudaMemcpyAsync(ids, b + L.ids, n * 4, cudaMemcpyDeviceToDevice, st);
    if (wts && e == cudaSuccess)
        e = cudaMemcpyAsync(wts, b + L.wts, n * 4, cudaMemcpyDeviceToDevice, st);
    if (uni && e == cudaSuccess)
        e = cudaMemcpyAsync(uni, b + L.uni, sizeof(moe_union_table), cudaMemcpyDeviceToDevice, st);
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "cudaMemcpyAsync: %s", cudaGetErrorString(e));
    return ok();
}

moe_status moe_read_device_status(void *ws, size_t ws_bytes, int *code, void *stream) {
    if (!ws || !aligned(ws, 256) || ws_bytes < sizeof(WsHeader))
        return fail(MOE_ERR_WORKSPACE, "workspace NULL, misaligned or too small");
    if (!code) return fail(MOE_ERR_INVALID_ARG, "code is NULL");
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    WsHeader h;
    cudaError_t e = cudaStreamSynchronize(st);
    if (e == cudaSuccess) e = cudaMemcpy(&h, ws, sizeof h, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemset(ws, 0, 2 * sizeof(uint32_t));
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
    *code = (int)h.status;
    if (h.status)
        return fail(MOE_ERR_DEVICE_STATUS, "device status %u (detail %u)", h.status,
                    h.status_info);
    return ok();
}

}  // extern "C"
