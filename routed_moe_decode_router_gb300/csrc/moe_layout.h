// moe_layout.h -- workspace layout and kernel parameter blocks shared by the
// host launch code and the kernels of the routed MoE library.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "../../include/moe_router.h"

namespace moe {

// One pass of the layer kernel: a sub-chunk of at most 8 rows and 64 ids.
constexpr int kMaxRows = MOE_CHUNK_ROWS;
constexpr int kMaxIds = MOE_CHUNK_IDS;
constexpr int kSharedEntry = kMaxIds;    // pointer-table slot of the shared expert
constexpr int kEntries = kMaxIds + 1;
// One call: up to 32 rows and 256 ids (several sub-chunks).
constexpr int kCallRows = MOE_MAX_ROWS;
constexpr int kCallIds = MOE_MAX_IDS;

// The union of one sub-chunk, as the layer kernel keeps it in shared memory
// (positions p = row * top_k + slot of the sub-chunk).
struct ChunkUnion {
    int32_t num_union;
    int32_t rows;
    int32_t top_k;
    int32_t per_row_mode;
    int32_t expert[kMaxIds];
    uint8_t rowmask[kMaxIds];
    uint8_t slot2u[kMaxIds];
    uint8_t uslot[kMaxIds][kMaxRows];
};
constexpr int kTileRows = 16;            // output rows of one MMA tile (M)
constexpr int kOutTile = 32;             // output rows of a down unit / blend tile
constexpr int kChunk = 128;              // inputs per compute-warp chunk
constexpr int kConsumerWarps = 8;        // compute warps of the layer kernel
constexpr int kRouteWarps = 8;
// Layer kernel block: 8 compute warps, 2 epilogue warps, 1 producer warp.
constexpr int kLayerBlockThreads = (kConsumerWarps + 3) * 32;
// CTAs of a t-layout launch whose partial outputs the workspace holds (one
// per SM of the device: at most 256).
constexpr int kMaxTCtas = 256;

// Status word and counters at the start of the workspace (256 bytes).
//
// Every launch of the layer kernel adds exactly one to launch_ticket per CTA,
// first thing after its dependency wait, so launch n (counted from the last
// zeroing of the workspace) reads tickets n*G .. n*G + G-1.  Launch n runs
// its grid barriers on bar_count[n & 1] and zeroes bar_count[(n + 1) & 1]
// for launch n + 1.  A launch whose barrier wait ran out leaves its own
// counter misaligned, but the next launch uses the other, freshly zeroed
// one, so the workspace needs no re-initialisation after a timeout.
struct WsHeader {
    uint32_t status;        // first MOE_DEV_* fault recorded (0 = none)
    uint32_t status_info;   // detail of that fault (offending id / unit)
    uint32_t route_ticket;  // last-block ticket of the route kernel
    uint32_t pad0;
    unsigned long long launch_ticket;   // CTAs of all layer launches so far
    unsigned long long bar_count[2];    // grid barriers of even / odd launches
    uint32_t pad[54];
};
static_assert(sizeof(WsHeader) == 256, "header size");

// Device pointer table entry of one union expert (or the shared expert):
// gate, up and down NVFP4 matrices.
struct PtrEntry {
    const uint8_t *packed[3];
    const uint8_t *scales[3];
    float scale2[3];
    int32_t expert;         // -1 marks an entry the kernels must skip
};
static_assert(sizeof(PtrEntry) == 64, "pointer entry size");

inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// Byte offsets of every workspace region for one configuration.  The ids,
// weights, union table and pointer table are sized for a whole call (32
// rows, 256 ids); the logits and the intermediate activations for one
// sub-chunk (8 rows), which the sub-chunks of a call reuse in turn.  One
// workspace serves every row count.
struct WsLayout {
    size_t header, ids, wts, logits, gate_val, uni, ptrs, hbuf, ybuf, ysbuf, ypart, total;
    int inter_max;          // max(I, Is): row stride of the h buffer

    static WsLayout make(const moe_config &c) {
        WsLayout L{};
        size_t o = 0;
        L.header = o;   o = align256(o + sizeof(WsHeader));
        // forward_token_major.rs scratch order: ids, then routing weights.
        L.ids = o;      o += sizeof(int32_t) * (size_t)kCallIds;
        L.wts = o;      o = align256(o + sizeof(float) * (size_t)kCallIds);
        L.logits = o;   o = align256(o + sizeof(float) * (size_t)kMaxRows * c.num_experts);
        L.gate_val = o; o = align256(o + sizeof(float) * kMaxRows);
        L.uni = o;      o = align256(o + sizeof(moe_union_table));
        L.ptrs = o;     o = align256(o + sizeof(PtrEntry) * (kCallIds + 1));
        L.inter_max = c.moe_inter;
        if (c.has_shared && c.shared_inter > L.inter_max) L.inter_max = c.shared_inter;
        L.hbuf = o;     o = align256(o + 2 * (size_t)kEntries * kMaxRows * L.inter_max);
        L.ybuf = o;     o = align256(o + sizeof(float) * (size_t)kMaxIds * c.hidden);
        L.ysbuf = o;    o = align256(o + sizeof(float) * (size_t)kMaxRows * c.hidden);
        // t layout: one partial output row per CTA
        L.ypart = o;    o = align256(o + (c.t_layout ? sizeof(float) * (size_t)kMaxTCtas * c.hidden : 0));
        L.total = o;
        return L;
    }
};

// Pointers into one workspace.
struct WsPtrs {
    WsHeader *hdr;
    int32_t *ids;
    float *wts;
    float *logits;
    float *gate_val;
    moe_union_table *uni;   // the call's union (all its rows)
    PtrEntry *ptrs;         // [kCallIds + 1]: union entries, the shared expert last
    uint16_t *hbuf;   // bf16 [kEntries][kMaxRows][inter_max]
    float *ybuf;      // fp32 [kMaxIds][H]: position p = row * top_k + slot
    float *ysbuf;     // fp32 [kMaxRows][H]: shared expert output
    float *ypart;     // fp32 [kMaxTCtas][H]: per-CTA partial outputs (t layout)
    int inter_max;
};

inline WsPtrs ws_ptrs(void *ws, const WsLayout &L) {
    char *b = static_cast<char *>(ws);
    WsPtrs p;
    p.hdr = reinterpret_cast<WsHeader *>(b + L.header);
    p.ids = reinterpret_cast<int32_t *>(b + L.ids);
    p.wts = reinterpret_cast<float *>(b + L.wts);
    p.logits = reinterpret_cast<float *>(b + L.logits);
    p.gate_val = reinterpret_cast<float *>(b + L.gate_val);
    p.uni = reinterpret_cast<moe_union_table *>(b + L.uni);
    p.ptrs = reinterpret_cast<PtrEntry *>(b + L.ptrs);
    p.hbuf = reinterpret_cast<uint16_t *>(b + L.hbuf);
    p.ybuf = reinterpret_cast<float *>(b + L.ybuf);
    p.ysbuf = reinterpret_cast<float *>(b + L.ysbuf);
    p.ypart = reinterpret_cast<float *>(b + L.ypart);
    p.inter_max = L.inter_max;
    return p;
}

// Parameters of the route kernel (router + top-k) for one sub-chunk of at
// most 8 rows, the call's rows row_base .. row_base + rows - 1.
struct RouteParams {
    int H, E, k, rows, row_base;
    int scoring, norm, router_fmt, has_shared, shared_gated, per_row_mode;
    float rsf;
    const uint16_t *x;
    const uint16_t *router_bf16;
    moe_nvfp4 router_fp4;
    const float *bias;
    const uint16_t *sh_vec;
    moe_expert_table gate, up, down;
    moe_nvfp4 sh_gate, sh_up, sh_down;
    WsPtrs ws;
    int32_t *ids_out;       // optional copies for moe_route (may be null)
    float *wts_out;
    float *logits_out;
};

// Parameters of the union kernel (moe_union, and calls of several
// sub-chunks): up to kCallIds ids.
struct UnionParams {
    int E, k, rows, per_row_mode, has_tables, has_shared, has_scales;
    const int32_t *ids;
    moe_expert_table gate, up, down;
    moe_nvfp4 sh_gate, sh_up, sh_down;
    WsPtrs ws;
    moe_union_table *out;
};

// Parameters of the persistent layer kernel for one sub-chunk of at most 8
// rows, the call's rows row_base .. row_base + rows - 1.  publish_union: the
// call has only this sub-chunk, so its union is the call's (written to the
// workspace for moe_read_routing).
// Whether a down unit of a layer-kernel instantiation (expert format fmt,
// MC_D B-fragment chunks per warp) can need K-parts, i.e. an FP8 / BF16
// down tile of 32 rows that does not fit two ring slots: BF16 from 13
// chunks (MC_D >= 2), FP8 from 26 chunks (MC_D = 4).  The other
// instantiations carry no K-part code.
__host__ __device__ constexpr bool down_parts_possible(int fmt, int mc_d) {
    return fmt == 2 ? mc_d >= 2 : (fmt == 1 && mc_d == 4);
}

struct LayerParams {
    int H, E, k, rows, I, Is;
    int row_base, publish_union;
    int scoring, norm, router_fmt, has_shared, shared_gated, per_row_mode;
    float rsf;
    int stages;
    uint32_t slot_bytes;
    int down_rows;          // output rows of a down unit: 32, or 64 (wide units)
    int down_split;         // 32-row units whose 8, 12 or 16 chunks go four to a tile
    int gu_halves;          // 2: BF16 gate/up tiles in two K-halves (one ring slot each)
    int down_pc;            // 128-input chunks of a down unit per ring slot (FP8 / BF16
                            // down units of more chunks come in K-parts, one slot each)
    const uint16_t *x;
    uint16_t *out;
    const uint16_t *router_bf16;
    moe_nvfp4 router_fp4;
    const float *bias;
    const uint16_t *sh_vec;
    moe_expert_table gate, up, down;
    moe_nvfp4 sh_gate, sh_up, sh_down;
    WsPtrs ws;
};

}  // namespace moe
