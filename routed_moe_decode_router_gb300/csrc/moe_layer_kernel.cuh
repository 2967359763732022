// moe_layer_kernel.cuh -- the whole routed MoE layer as one persistent kernel.
//
// One CTA per SM (every CTA resident at once): 8 compute warps, 2 epilogue
// warps (cross-warp reductions and output stores; they take alternate units,
// each fed through its own buffer of partial sums behind mbarriers, so the
// compute warps rarely wait for an epilogue) and 1 producer warp (bulk
// copies).  Phases:
//   A  router: the E router rows (plus the shared-expert gate vector as row
//      E) are spread over the CTAs; each row's dot products for all token
//      rows are split over the compute warps (forward_token_major.rs:
//      dense_gemm / w4a16_gemm).  Meanwhile the producer stages this CTA's
//      first shared-expert gate/up tiles, which need no routing.
//   -  grid barrier (all logits written)
//   B  every CTA computes the top-k of every row and the union itself, from
//      the logits in L2 -- the same result in every CTA, so no second
//      exchange is needed (page "Function forward_moe", RETRACTED and WIDENED
//      notes: up to 64 ids, de-duplicated by pairwise comparison in one
//      block, never sorted or sent to the host); the producer then
//      fetches the union experts' pointer entries.
//   C  gate+up sweep: units = 16-row tiles of an entry's gate and up
//      matrices (shared expert first, then the union experts), CTA b takes
//      units b, b + G, ...; h = bf16(silu(g) * v) to the workspace
//      (moe_expert_gate_up_shared_prefill).
//   -  grid barrier (every h written); the producer keeps streaming down
//      tiles through it
//   D  down sweep: units = 32-row tiles of an entry's down matrix, CTA b
//      takes a contiguous range (h fragments stay in registers per entry);
//      y (fp32) per (row, slot) to the workspace
//      (moe_expert_silu_down_shared_prefill).
//   -  grid barrier (every y written)
//   E  blend, spread over the CTAs by (32-row output tile, token row):
//        out[r][o] = bf16( sum_{slot<k} w[r][slot] * y[r][slot][o] + g_r * ys[r][o] )
//      in slot order (moe_weighted_sum_blend_prefill).
//
// Weight tiles (contiguous 16 x K/2 packed + 16 x K/16 scale bytes) move by
// bulk (TMA) copies into a ring of shared-memory slots behind mbarriers with
// an evict-first L2 policy; gate and up of one unit occupy two slots, a down
// unit one.  The MMA is mma.sync m16n8k16 (f16 x f16 -> fp32) with the NVFP4
// weights unpacked to f16 in registers and the token rows as the 8 columns.
//
// With the down projections in the t layout (input-major, one row per
// intermediate index; one token row per launch) the layer is fused instead:
// each gate+up unit also streams its 16 rows of the transposed down matrix
// (a third ring slot), the compute warps apply them to the unit's h as soon
// as the epilogue warp has formed it, and each CTA keeps a partial sum of
// every output; after phase C one grid barrier, then CTA b adds up its slice
// of the outputs over all CTAs' partials in CTA order.  Phases D and E and
// grid barrier 3 do not exist in this form.
//
// Every wait is bounded (ring waits, the grid barriers); a wait that runs
// out records MOE_DEV_WAIT_TIMEOUT, and the CTA skips the rest of its work.
#pragma once
#include <cuda_runtime.h>

#include "moe_blocks.cuh"

// Phase marks and cycle accumulators: no-ops unless the library is built with
// MOE_TRACE, which must then provide moe_trace_mark(cta, mark) (a per-CTA
// timestamp store) and moe_trace_add(cta, slot, cycles).
#ifdef MOE_TRACE
__device__ void moe_trace_mark(int cta, int mark);
__device__ void moe_trace_add(int cta, int slot, long long cycles);
#define MOE_PHASE_MARK(cond, i) \
    do {                        \
        if (cond) moe_trace_mark(blockIdx.x, (i)); \
    } while (0)
#define MOE_TIC(v) const long long v = clock64()
#define MOE_TOC(cond, i, v) \
    do {                    \
        if (cond) moe_trace_add(blockIdx.x, (i), clock64() - (v)); \
    } while (0)
#else
#define MOE_PHASE_MARK(cond, i) \
    do {                        \
    } while (0)
#define MOE_TIC(v) \
    do {           \
    } while (0)
#define MOE_TOC(cond, i, v) \
    do {                    \
    } while (0)
#endif

namespace moe {

constexpr int kRouterRowsPerPass = 4;     // router rows of one CTA handled together
constexpr int kMaxSegs = MOE_MAX_HIDDEN / 256;
constexpr int kRed = 2;                   // partial-sum buffers between compute and epilogue
constexpr int kEpiWarp = kConsumerWarps;        // warp 8: first epilogue warp (and the union)
constexpr int kProdWarp = kConsumerWarps + 1;   // warp 9: bulk-copy producer
constexpr int kEpiWarp2 = kConsumerWarps + 2;   // warp 10: second epilogue warp
constexpr int kEpiWarps = 2;                    // epilogue warp e takes units ui with ui % 2 == e
constexpr int kLayerThreads = kLayerBlockThreads;
constexpr int kComputeAndEpi = (kConsumerWarps + kEpiWarps) * 32;
static_assert(kRed == kEpiWarps, "each epilogue warp owns one partial-sum buffer");

struct LayerSmem {
    float red[kRed][kConsumerWarps][256];       // compute warps' partial sums
    float rpart[kRouterRowsPerPass][kMaxSegs][kMaxRows];   // router partial dots
    ChunkUnion uni;
    PtrEntry ptrs[kEntries];
    int32_t ids[kMaxIds];
    float wts[kMaxIds];
    float gate_val[kMaxRows];
    uint32_t umask[kMaxIds];
    uint64_t red_full[kRed];                    // partials ready (8 compute-warp arrivals)
    uint64_t red_empty[kRed];                   // partials consumed (1 epilogue arrival)
    // t layout: the h values of a gate+up unit, handed from the epilogue
    // warp that formed them to the compute warps (one slot per epilogue warp)
    float hsm[kEpiWarps][kTileRows];
    uint64_t h_full[kEpiWarps];                 // h written (1 epilogue arrival)
    uint64_t h_empty[kEpiWarps];                // h read (8 compute-warp arrivals)
    unsigned long long *bar;                    // this launch's grid-barrier counter
    int abort;
};

constexpr size_t kLayerSmemFixed = (sizeof(LayerSmem) + 127) & ~size_t(127);

// Raw router weights of row `row` (E = the shared-expert gate vector) at the
// 8 inputs h0..h0+7: a uint4 of bf16 values, or (NVFP4) the packed word in
// .x and the E4M3 scale byte in .y.  Loads only, so that several rows' loads
// can be in flight before any is used.
__device__ __forceinline__ uint4 router_raw(const LayerParams &p, int row, int h0) {
    const int H = p.H;
    if (row == p.E || p.router_fmt == MOE_ROUTER_BF16) {
        const uint16_t *src = (row == p.E) ? p.sh_vec + h0 : p.router_bf16 + (size_t)row * H + h0;
        return ld_nc_v4(src);
    }
    uint4 r;
    r.x = *reinterpret_cast<const uint32_t *>(p.router_fp4.packed + (size_t)row * (H / 2) + h0 / 2);
    r.y = p.router_fp4.scales[(size_t)row * (H / 16) + h0 / 16];
    r.z = r.w = 0u;
    return r;
}

// The 8 weights of router_raw as fp32 (NVFP4: e2m1 * e4m3; scale2 comes later).
__device__ __forceinline__ void router_decode(const LayerParams &p, int row, uint4 v, float (&w)[8]) {
    if (row == p.E || p.router_fmt == MOE_ROUTER_BF16) {
        w[0] = bf16_lo(v.x); w[1] = bf16_hi(v.x); w[2] = bf16_lo(v.y); w[3] = bf16_hi(v.y);
        w[4] = bf16_lo(v.z); w[5] = bf16_hi(v.z); w[6] = bf16_lo(v.w); w[7] = bf16_hi(v.w);
    } else {
        const uint32_t sh = e4m3x2_to_f16x2(v.y);
        const float sc = __low2float(*reinterpret_cast<const __half2 *>(&sh));
        uint32_t hq[4];
        e2m1x8_to_f16x2(v.x, hq);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __half2 qv = *reinterpret_cast<const __half2 *>(&hq[i]);
            w[2 * i] = __low2float(qv) * sc;
            w[2 * i + 1] = __high2float(qv) * sc;
        }
    }
}

// MC_GU / MC_D: B-fragment chunks per compute warp in the gate+up / down
// phases; TK: the top-k class of the router width (0: E <= 128, 1: <= 256,
// 2: <= 512, 3: <= 1024), so each instantiation holds one top-k variant;
// GV: the one-row CUDA-core GEMV variant of the expert projections
// (chunk_gemv) instead of the tensor-core MMA (chunk_mma); TL: the fused
// one-row form for down projections in the t layout (MC_D unused); FMT: the
// expert format (0 NVFP4, 1 FP8, 2 BF16; the GEMV variant and the t layout
// exist for NVFP4 only); KP: the FP8 / BF16 instantiations whose down units
// come in K-parts (down tiles beyond the ring), compiled apart from the
// others (moe_layer_tk*_kp.cu) so that their code does not share a module
// with the instantiations that never need it.
template <int MC_GU, int MC_D, int TK, bool GV, bool TL, int FMT = 0, bool KP = false>
__global__ void __launch_bounds__(kLayerThreads, 1) moe_layer_kernel(const LayerParams p) {
    static_assert(FMT == 0 || (!GV && !TL), "GEMV variant and t layout: NVFP4 experts only");
    static_assert(!KP || down_parts_possible(FMT, MC_D), "K-parts: FP8 / BF16 with enough chunks per warp");
    constexpr bool kDownParts = KP;
    // one-row form with 4 chunks per warp (hidden 3200 .. 4096, a ring of 5
    // to 7 slots): each unit's gate slot is released before its up slot is
    // waited for, which keeps one more slot in flight; the other
    // instantiations multiply gate and up chunks interleaved (two independent
    // chains), which the multi-row sweeps need
    constexpr bool kGateFirst = TL && MC_GU == 4;
    extern __shared__ __align__(128) uint8_t smem[];
    LayerSmem &sm = *reinterpret_cast<LayerSmem *>(smem);
    uint8_t *ring = smem + kLayerSmemFixed;
    uint64_t *full = reinterpret_cast<uint64_t *>(ring + (size_t)p.stages * p.slot_bytes);
    uint64_t *empty = full + p.stages;
    volatile int *abort = &sm.abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = gridDim.x, b = blockIdx.x, S = p.stages;
    const int H = p.H, E = p.E, k = p.k;
    const int It = p.I / kTileRows;
    const int St = p.has_shared ? p.Is / kTileRows : 0;
    const int Ho = H / kOutTile;                 // 32-row output tiles (blend)
    // down units: DR output rows each (32, or 64 when every entry's
    // intermediate is 2 or 4 chunks wide: "wide" units, whose chunks and
    // 16-row tiles are spread over all eight compute warps)
    const int DR = p.down_rows, Hd = H / DR;
    const bool wide = DR == 2 * kOutTile;
    // "split" 32-row units (down_split): warp w multiplies tile w / 4 of the
    // unit at chunks w % 4 + 4 m, so an intermediate of 8, 12 or 16 chunks
    // gives every warp the same work and the epilogue four partials a tile
    const bool split = p.down_split != 0;
    const int Sd = p.has_shared ? Hd : 0;
    const bool is_comp = warp < kConsumerWarps;
    const bool is_epi = warp == kEpiWarp || warp == kEpiWarp2;
    const int epi_idx = warp == kEpiWarp2 ? 1 : 0;
    const bool is_prod = warp == kProdWarp;
    const bool gate_row = p.has_shared && p.shared_gated;
    const int nrow = E + (gate_row ? 1 : 0);
    const uint32_t gu_pk = kTileRows * fmt_row_bytes<FMT>(H);
    const uint32_t gu_sc = kTileRows * fmt_scale_row_bytes<FMT>(H);
    WsHeader *hdr = p.ws.hdr;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        for (int r = 0; r < kRed; ++r) {
            mbar_init(&sm.red_full[r], kConsumerWarps);
            mbar_init(&sm.red_empty[r], 1);
        }
        for (int r = 0; r < kEpiWarps; ++r) {
            mbar_init(&sm.h_full[r], 1);
            mbar_init(&sm.h_empty[r], kConsumerWarps);
        }
        fence_mbar_init();
        sm.abort = 0;
    }
    __syncthreads();
    MOE_PHASE_MARK(tid == 0, 0);

    // ---------------- producer: slot issue helpers (lane 0 only) ----------------
    uint64_t pol = 0;
    int pi = 0;   // slots issued
    auto acquire = [&](int i) -> bool {
        if (i < S) return !*abort;
        return ring_wait(&empty[i % S], ((i / S) - 1) & 1, abort, hdr, 0x100000u + (uint32_t)i);
    };
    auto issue_pair = [&](const uint8_t *pk, const uint8_t *sc, uint32_t pkb, uint32_t scb) {
        const int s = pi % S;
        uint8_t *st = ring + (size_t)s * p.slot_bytes;
        mbar_arrive_expect_tx(&full[s], pkb + scb);
        bulk_g2s(st, pk, pkb, &full[s], pol);
        if (scb) bulk_g2s(st + pkb, sc, scb, &full[s], pol);   // FP8 / BF16: no block scales
        ++pi;
    };
    // n rows of seg bytes at a source stride into one slot
    auto issue_rows = [&](const uint8_t *src, uint32_t stride, uint32_t seg, int n) {
        const int s = pi % S;
        uint8_t *st = ring + (size_t)s * p.slot_bytes;
        mbar_arrive_expect_tx(&full[s], seg * (uint32_t)n);
        for (int r = 0; r < n; ++r)
            bulk_g2s(st + (size_t)r * seg, src + (size_t)r * stride, seg, &full[s], pol);
        ++pi;
    };
    auto issue_empty = [&]() -> bool {
        if (!acquire(pi)) return false;
        mbar_arrive(&full[pi % S]);
        ++pi;
        return true;
    };
    // gate+up unit j (16 rows): a gate slot, then an up slot; in the t
    // layout also a slot with the unit's 16 rows of the transposed down
    // matrix (16 x H/2 packed bytes, then the H scales of that block).
    // BF16 gate/up tiles too large for the ring come in two K-halves: a unit
    // is then gate half 0, up half 0, gate half 1, up half 1 (a half tile is
    // 16 row segments of H bytes, one bulk copy each).
    const int ghalves = (FMT == 2) ? p.gu_halves : 1;
    const int unit_slots = TL ? 3 : 2 * ghalves;
    const uint32_t dt_pk = kTileRows * H / 2, dt_sc = H;
    auto issue_gu = [&](int j) -> bool {
        const uint8_t *gp, *gs, *upk, *us, *dp = nullptr, *ds = nullptr;
        if (j < St) {
            gp = p.sh_gate.packed + (size_t)j * gu_pk;
            gs = p.sh_gate.scales + (size_t)j * gu_sc;
            upk = p.sh_up.packed + (size_t)j * gu_pk;
            us = p.sh_up.scales + (size_t)j * gu_sc;
            if (TL) {
                dp = p.sh_down.packed + (size_t)j * dt_pk;
                ds = p.sh_down.scales + (size_t)j * dt_sc;
            }
        } else {
            const PtrEntry &e = sm.ptrs[(j - St) / It];
            const int tile = (j - St) % It;
            if (e.expert < 0) {
                bool ok2 = true;
                for (int i = 0; i < unit_slots; ++i) ok2 = ok2 && issue_empty();
                return ok2;
            }
            gp = e.packed[0] + (size_t)tile * gu_pk;
            gs = e.scales[0] + (size_t)tile * gu_sc;
            upk = e.packed[1] + (size_t)tile * gu_pk;
            us = e.scales[1] + (size_t)tile * gu_sc;
            if (TL) {
                dp = e.packed[2] + (size_t)tile * dt_pk;
                ds = e.scales[2] + (size_t)tile * dt_sc;
            }
        }
        if (FMT == 2 && ghalves == 2) {
            const uint32_t row = fmt_row_bytes<FMT>(H), half = row / 2;
            for (int h = 0; h < 2; ++h) {
                if (!acquire(pi)) return false;
                issue_rows(gp + h * half, row, half, kTileRows);
                if (!acquire(pi)) return false;
                issue_rows(upk + h * half, row, half, kTileRows);
            }
            return true;
        }
        if (!acquire(pi)) return false;
        issue_pair(gp, gs, gu_pk, gu_sc);
        if (!acquire(pi)) return false;
        issue_pair(upk, us, gu_pk, gu_sc);
        if (TL) {
            if (!acquire(pi)) return false;
            issue_pair(dp, ds, dt_pk, dt_sc);
        }
        return true;
    };

    int pj = b;   // next gate+up unit of this CTA
    if (is_prod && lane == 0) {
        pol = l2_evict_first_policy();
        while (pj < St && pi + unit_slots <= S) {
            issue_gu(pj);
            pj += G;
        }
        MOE_PHASE_MARK(true, 11);
    }
    // L2 prefetch of this CTA's router rows and of the expert tables
    if (is_comp && lane == 0) {
        for (int row = b + G * warp; row < nrow; row += G * kConsumerWarps) {
            const void *src;
            uint32_t bytes;
            if (row == E) {
                src = p.sh_vec;
                bytes = H * 2;
            } else if (p.router_fmt == MOE_ROUTER_BF16) {
                src = p.router_bf16 + (size_t)row * H;
                bytes = H * 2;
            } else {
                src = p.router_fp4.packed + (size_t)row * (H / 2);
                bytes = H / 2;
            }
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes)
                         : "memory");
        }
    }
    if (b < 3 && warp == 0) {
        const moe_expert_table &t = b == 0 ? p.gate : (b == 1 ? p.up : p.down);
        for (int off = lane * 128; off < E * 8; off += 32 * 128) {
            asm volatile("prefetch.global.L2 [%0];" ::"l"((const char *)t.packed + off));
            asm volatile("prefetch.global.L2 [%0];" ::"l"((const char *)t.scales + off));
        }
        for (int off = lane * 128; off < E * 4; off += 32 * 128)
            asm volatile("prefetch.global.L2 [%0];" ::"l"((const char *)t.scale2 + off));
    }
    pdl_trigger();
    pdl_wait();
    // launch ticket (the second epilogue warp is idle in phase A): this
    // launch's barrier counter, and the next launch's counter zeroed
    if (warp == kEpiWarp2 && lane == 0) {
        const unsigned long long n = atomicAdd(&hdr->launch_ticket, 1ULL) / (unsigned)G;
        sm.bar = &hdr->bar_count[n & 1];
        if (b == 0) hdr->bar_count[(n + 1) & 1] = 0ULL;
    }
    MOE_PHASE_MARK(tid == 0, 1);

    // ---------------- phase A: router rows ----------------
    // This CTA's rows are b, b + G, ... (at most kRouterRowsPerPass per
    // pass).  Compute warp w takes the 256-input segments w, w + 8, ...: it
    // loads the token rows' inputs of its segment once, then the weights of
    // every row of the pass, all before the first use, so one memory latency
    // covers the pass.  Partial sums are added in segment order.
    // (the one-row form's instantiations are compiled for one token row)
    constexpr int RR = TL ? 1 : kMaxRows;
    if (is_comp) {
        const int my_rows = b < nrow ? (nrow - b + G - 1) / G : 0;
        const int nseg = (H + 255) / 256;
        for (int r0 = 0; r0 < my_rows; r0 += kRouterRowsPerPass) {
            const int nr = min(kRouterRowsPerPass, my_rows - r0);
            for (int seg = warp; seg < nseg; seg += kConsumerWarps) {
                const int h0 = seg * 256 + lane * 8;
                const bool live = h0 < H;   // H is a multiple of 128, not always of 256
                const int hc = live ? h0 : 0;
                // every load first, from clamped addresses; unused values are zeroed after
                uint4 xv[RR];
#pragma unroll
                for (int r = 0; r < RR; ++r)
                    if (r < p.rows) xv[r] = ld_cg_v4(p.x + (size_t)r * H + hc);
                uint4 rv[kRouterRowsPerPass];
#pragma unroll
                for (int ri = 0; ri < kRouterRowsPerPass; ++ri)
                    rv[ri] = router_raw(p, b + (r0 + min(ri, nr - 1)) * G, hc);
#pragma unroll
                for (int r = 0; r < RR; ++r)
                    if (!live || r >= p.rows) xv[r] = make_uint4(0u, 0u, 0u, 0u);
                float wv[kRouterRowsPerPass][8];
#pragma unroll
                for (int ri = 0; ri < kRouterRowsPerPass; ++ri) {
                    router_decode(p, b + (r0 + min(ri, nr - 1)) * G, rv[ri], wv[ri]);
                    if (!live || ri >= nr) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) wv[ri][i] = 0.f;
                    }
                }
                if (!TL && (TK >= 2 || (TK == 1 && p.rows >= 2))) {
                    // wide routers (E > 256), or two or more token rows at
                    // E <= 256: the 32 (router row, token row) lane partials
                    // by one reduce-scatter butterfly (31 shuffles instead of
                    // up to 160).
                    // Value v = ri * 8 + r; at offset o a lane keeps the half
                    // of its values whose bit o matches its own lane bit and
                    // adds the partner's copy of it, so the pairs are those of
                    // the per-value butterfly (same bits) and lane v ends
                    // with value v.
                    float a[kRouterRowsPerPass * kMaxRows];
#pragma unroll
                    for (int ri = 0; ri < kRouterRowsPerPass; ++ri)
#pragma unroll
                        for (int r = 0; r < kMaxRows; ++r) {
                            const uint4 x4 = xv[min(r, RR - 1)];
                            float t = 0.f;
                            t = fmaf(bf16_lo(x4.x), wv[ri][0], t);
                            t = fmaf(bf16_hi(x4.x), wv[ri][1], t);
                            t = fmaf(bf16_lo(x4.y), wv[ri][2], t);
                            t = fmaf(bf16_hi(x4.y), wv[ri][3], t);
                            t = fmaf(bf16_lo(x4.z), wv[ri][4], t);
                            t = fmaf(bf16_hi(x4.z), wv[ri][5], t);
                            t = fmaf(bf16_lo(x4.w), wv[ri][6], t);
                            t = fmaf(bf16_hi(x4.w), wv[ri][7], t);
                            a[ri * kMaxRows + r] = (r < p.rows) ? t : 0.f;
                        }
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) {
                        const bool up = (lane & o) != 0;
#pragma unroll
                        for (int i = 0; i < o; ++i) {
                            const float keep = up ? a[o + i] : a[i];
                            const float give = up ? a[i] : a[o + i];
                            a[i] = keep + __shfl_xor_sync(0xffffffffu, give, o);
                        }
                    }
                    const int ri = lane / kMaxRows, r = lane % kMaxRows;
                    if (ri < nr && r < p.rows) sm.rpart[ri][seg][r] = a[0];
                } else {
#pragma unroll
                    for (int ri = 0; ri < kRouterRowsPerPass; ++ri) {
                        if (ri >= nr) break;
#pragma unroll
                        for (int r = 0; r < RR; ++r) {
                            if (r >= p.rows) break;
                            const uint4 x4 = xv[r];
                            float a = 0.f;
                            a = fmaf(bf16_lo(x4.x), wv[ri][0], a);
                            a = fmaf(bf16_hi(x4.x), wv[ri][1], a);
                            a = fmaf(bf16_lo(x4.y), wv[ri][2], a);
                            a = fmaf(bf16_hi(x4.y), wv[ri][3], a);
                            a = fmaf(bf16_lo(x4.z), wv[ri][4], a);
                            a = fmaf(bf16_hi(x4.z), wv[ri][5], a);
                            a = fmaf(bf16_lo(x4.w), wv[ri][6], a);
                            a = fmaf(bf16_hi(x4.w), wv[ri][7], a);
#pragma unroll
                            for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
                            if (lane == 0) sm.rpart[ri][seg][r] = a;
                        }
                    }
                }
            }
            named_bar(1, kConsumerWarps * 32);
            for (int t = tid; t < nr * p.rows; t += kConsumerWarps * 32) {
                const int ri = t / p.rows, r = t % p.rows;
                const int row = b + (r0 + ri) * G;
                float v = 0.f;
                for (int seg = 0; seg < nseg; ++seg) v += sm.rpart[ri][seg][r];
                if (row == E) {
                    p.ws.gate_val[r] = 1.f / (1.f + expf(-v));
                } else {
                    if (p.router_fmt == MOE_ROUTER_NVFP4) v *= p.router_fp4.scale2;
                    p.ws.logits[(size_t)r * E + row] = v;
                }
            }
            named_bar(1, kConsumerWarps * 32);
        }
    }
    __syncthreads();
    MOE_PHASE_MARK(tid == 0, 2);
    if (tid == 0) grid_arrive_wait(sm.bar, G, abort, hdr, 1u);
    __syncthreads();
    MOE_PHASE_MARK(tid == 0, 3);

    // ---------------- phase B: top-k and union, in every CTA ----------------
    // One warp per token row selects its experts; then the epilogue warp
    // builds the union and the union experts' pointer entries while the
    // compute warps load their token-row fragments, and publishes both
    // through named barrier 4.
    if (warp == kEpiWarp && lane < kMaxRows)
        sm.gate_val[lane] = !p.has_shared ? 0.f : (gate_row ? ld_cg(p.ws.gate_val + lane) : 1.f);
    MOE_TIC(t_topk);
    if (warp < p.rows)
        warp_topk_row_tk<TK>(p.ws.logits + (size_t)warp * E, p.bias, E, k, p.scoring, p.norm,
                             p.rsf, sm.ids + warp * k, sm.wts + warp * k, lane);
    MOE_TOC(tid == 0, 16, t_topk);
    __syncthreads();
    if (warp == kEpiWarp) {
        MOE_TIC(t_union);
        UnionSrc src{E,      k,      p.rows,  p.per_row_mode, 1,       p.has_shared, FMT == 0,
                     p.gate, p.up,   p.down,  p.sh_gate,      p.sh_up, p.sh_down};
        if constexpr (TL)
            build_union_one_row(src, sm.ids, &sm.uni, sm.ptrs, hdr, lane);
        else
            build_union(src, sm.ids, sm.umask, &sm.uni, sm.ptrs, hdr, lane);
        __syncwarp();
        asm volatile("bar.arrive 4, %0;" ::"r"(kLayerThreads) : "memory");
        MOE_TOC(lane == 0, 17, t_union);
        MOE_PHASE_MARK(lane == 0, 4);
        if (b == 0) {   // publish the routing for moe_read_routing
            const int n = p.rows * k;
            for (int i = lane; i < n; i += 32) {
                p.ws.ids[p.row_base * k + i] = sm.ids[i];
                p.ws.wts[p.row_base * k + i] = sm.wts[i];
            }
            if (p.publish_union) {   // this sub-chunk is the whole call
                moe_union_table *g = p.ws.uni;
                uint4 *us = reinterpret_cast<uint4 *>(&g->uslot[0][0]);
                for (int i = lane; i < (int)(sizeof(g->uslot) / 16); i += 32)
                    us[i] = make_uint4(~0u, ~0u, ~0u, ~0u);
                __syncwarp();
                const int U = sm.uni.num_union;
                for (int u = lane; u < U; u += 32) {
                    g->expert[u] = sm.uni.expert[u];
                    g->rowmask[u] = sm.uni.rowmask[u];
#pragma unroll
                    for (int r = 0; r < kMaxRows; ++r) g->uslot[u][r] = sm.uni.uslot[u][r];
                }
                for (int i = lane; i < n; i += 32) g->slot2u[i] = sm.uni.slot2u[i];
                if (lane == 0) {
                    g->num_union = U;
                    g->rows = p.rows;
                    g->top_k = k;
                    g->per_row_mode = p.per_row_mode;
                }
            }
            if (lane < kMaxRows && !gate_row) p.ws.gate_val[lane] = sm.gate_val[lane];
        }
    } else if (is_prod || warp == kEpiWarp2) {
        named_bar(4, kLayerThreads);
    }
    // (the compute warps pass barrier 4 after loading their fragments)
    const uint32_t allrows = (1u << p.rows) - 1u;
    int U = 0, Tgu = 0, Td = 0, d_begin = 0, d_end = 0;
    auto sweep_layout = [&]() {
        U = sm.uni.num_union;
        Tgu = St + U * It;
        Td = Sd + U * Hd;
        d_begin = (int)((long long)b * Td / G);
        d_end = (int)((long long)(b + 1) * Td / G);
    };

    // ---------------- producer: pointer table, then every remaining slot ----------------
    if (is_prod) {
        sweep_layout();
        if (lane == 0) {
            bool ok = true;
            for (; ok && pj < Tgu; pj += G) ok = issue_gu(pj);
            for (int j = d_begin; !TL && ok && j < d_end; ++j) {
                const uint8_t *dp, *ds;
                int K;
                if (j < Sd) {
                    K = p.Is;
                    dp = p.sh_down.packed + (size_t)j * DR * fmt_row_bytes<FMT>(K);
                    ds = p.sh_down.scales + (size_t)j * DR * fmt_scale_row_bytes<FMT>(K);
                } else {
                    const PtrEntry &e = sm.ptrs[(j - Sd) / Hd];
                    const int tile = (j - Sd) % Hd;
                    if (e.expert < 0) {
                        ok = issue_empty();
                        if constexpr (kDownParts)
                            for (int c0 = p.down_pc; ok && c0 < p.I / kChunk; c0 += p.down_pc)
                                ok = issue_empty();
                        continue;
                    }
                    K = p.I;
                    dp = e.packed[2] + (size_t)tile * DR * fmt_row_bytes<FMT>(K);
                    ds = e.scales[2] + (size_t)tile * DR * fmt_scale_row_bytes<FMT>(K);
                }
                if constexpr (kDownParts) {
                    // FP8 / BF16 down unit in K-parts of down_pc chunks: DR
                    // row segments per slot
                    const int nch = K / kChunk;
                    if (nch > p.down_pc) {
                        for (int c0 = 0; ok && c0 < nch; c0 += p.down_pc) {
                            const int nc = min(p.down_pc, nch - c0);
                            if (!(ok = acquire(pi))) break;
                            issue_rows(dp + fmt_row_bytes<FMT>(c0 * kChunk), fmt_row_bytes<FMT>(K),
                                       fmt_row_bytes<FMT>(nc * kChunk), DR);
                        }
                        continue;
                    }
                }
                if (!(ok = acquire(pi))) break;
                issue_pair(dp, ds, DR * fmt_row_bytes<FMT>(K), DR * fmt_scale_row_bytes<FMT>(K));
            }
            MOE_PHASE_MARK(true, 10);
        }
        return;
    }

    if (is_epi) {
        // ---------------- epilogue warp ----------------
        // Everything a unit's epilogue needs except the partial sums (entry,
        // tile, scales, row mask, destination) is fetched before waiting for
        // them, and the eight warps' partials are loaded unconditionally and
        // summed with a select, so one shared-memory latency covers them.
        sweep_layout();
        int ui = 0;
        const int nwg = min(kConsumerWarps, H / kChunk);   // warps holding gate/up partials
        const int col = lane >> 2, rq = lane & 3;
        for (int j = b; j < Tgu; j += G, ++ui) {
            if ((ui & 1) != epi_idx) continue;
            const int rb = ui % kRed;
            int entry, tile;
            float s2g, s2u;
            uint32_t mask;
            bool live = true;
            if (j < St) {
                entry = kSharedEntry;
                tile = j;
                s2g = p.sh_gate.scale2;
                s2u = p.sh_up.scale2;
                mask = allrows;
            } else {
                entry = (j - St) / It;
                tile = (j - St) % It;
                live = sm.ptrs[entry].expert >= 0;
                s2g = sm.ptrs[entry].scale2[0];
                s2u = sm.ptrs[entry].scale2[1];
                mask = sm.uni.rowmask[entry];
            }
            live = live && ((mask >> col) & 1u);
            // lane: column col, rows 4 * rq .. + 3 of the 16-row tile
            const int off = partial_index(col, 4 * rq);
            MOE_TIC(t_ew);
            ring_wait(&sm.red_full[rb], (ui / kRed) & 1, abort, hdr, 0x200000u + (uint32_t)ui);
            MOE_TOC(lane == 0, 25, t_ew);
            MOE_TIC(t_ex);
            float4 ga[kConsumerWarps], ua[kConsumerWarps];
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                ga[w] = *reinterpret_cast<const float4 *>(&sm.red[rb][w][off]);
                ua[w] = *reinterpret_cast<const float4 *>(&sm.red[rb][w][128 + off]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.red_empty[rb]);   // the values are in registers
            float gs[4] = {0.f, 0.f, 0.f, 0.f}, us[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                const bool on = w < nwg;
                gs[0] += on ? ga[w].x : 0.f; gs[1] += on ? ga[w].y : 0.f;
                gs[2] += on ? ga[w].z : 0.f; gs[3] += on ? ga[w].w : 0.f;
                us[0] += on ? ua[w].x : 0.f; us[1] += on ? ua[w].y : 0.f;
                us[2] += on ? ua[w].z : 0.f; us[3] += on ? ua[w].w : 0.f;
            }
            if constexpr (TL) {
                // the unit's 16 h values (token row 0: lanes 0..3, rounded
                // to bf16) to this warp's slot, once the compute warps have
                // read its previous use
                float hf[4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    hf[i] = bf16_lo(f2bf16_rn(silu(gs[i] * s2g) * (us[i] * s2u)));
                const int hb = epi_idx;
                if (ui >= kEpiWarps)
                    ring_wait(&sm.h_empty[hb], ((ui / kEpiWarps) - 1) & 1, abort, hdr,
                              0x500000u + (uint32_t)ui);
                if (col == 0) {
                    const bool on = live && !*abort;
#pragma unroll
                    for (int i = 0; i < 4; ++i) sm.hsm[hb][4 * rq + i] = on ? hf[i] : 0.f;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.h_full[hb]);
            } else if (live && !*abort) {
                uint32_t hv[2];
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    float h2[2];
#pragma unroll
                    for (int z = 0; z < 2; ++z) {
                        const float gv = gs[2 * i + z] * s2g, uv = us[2 * i + z] * s2u;
                        h2[z] = silu(gv) * uv;
                    }
                    hv[i] = (uint32_t)f2bf16_rn(h2[0]) | ((uint32_t)f2bf16_rn(h2[1]) << 16);
                }
                *reinterpret_cast<uint2 *>(p.ws.hbuf +
                                           ((size_t)entry * kMaxRows + col) * p.ws.inter_max +
                                           tile * kTileRows + 4 * rq) = make_uint2(hv[0], hv[1]);
            }
            MOE_TOC(lane == 0, 26, t_ex);
        }
        if constexpr (TL) {
            // the compute warps finish the layer (partial outputs, grid
            // barrier, sum over the CTAs); the epilogue warps take the grid
            // barrier for them
            named_bar(3, kComputeAndEpi);   // every partial of this CTA stored
            MOE_PHASE_MARK(lane == 0 && epi_idx == 0, 13);
            if (lane == 0 && epi_idx == 0) grid_arrive_wait(sm.bar, G, abort, hdr, 2u);
            named_bar(3, kComputeAndEpi);   // every CTA's partials visible
            return;
        }
        // every h of this CTA is stored (both epilogue warps): grid barrier,
        // then release the compute warps
        named_bar(5, kEpiWarps * 32);
        MOE_PHASE_MARK(lane == 0 && epi_idx == 0, 13);
        if (lane == 0 && epi_idx == 0) grid_arrive_wait(sm.bar, G, abort, hdr, 2u);
        named_bar(5, kEpiWarps * 32);
        MOE_PHASE_MARK(lane == 0 && epi_idx == 0, 14);
        asm volatile("bar.arrive 2, %0;" ::"r"(kComputeAndEpi) : "memory");
        // lane: column col, rows 8 * (rq & 1) .. + 7 of MMA tile rq >> 1 (a
        // 32-row unit), or rows 4 * rq .. + 3 of each of the four MMA tiles
        // (a wide unit)
        const int half = rq >> 1, r0 = (rq & 1) * 8;
        for (int j = d_begin; j < d_end; ++j, ++ui) {
            if ((ui & 1) != epi_idx) continue;
            const int rb = ui % kRed;
            int entry, tile, K;
            uint32_t mask;
            float s2;
            bool live = true;
            if (j < Sd) {
                entry = kSharedEntry;
                tile = j;
                K = p.Is;
                mask = allrows;
                s2 = p.sh_down.scale2;
            } else {
                entry = (j - Sd) / Hd;
                tile = (j - Sd) % Hd;
                K = p.I;
                mask = sm.uni.rowmask[entry];
                live = sm.ptrs[entry].expert >= 0;
                s2 = sm.ptrs[entry].scale2[2];
            }
            live = live && ((mask >> col) & 1u);
            if (wide) {
                // tile t of the unit comes from the nch warps of tile group
                // t / tpg (chunks 0..nch-1, in that order), slot t % tpg
                const int nch = K / kChunk, tpg = nch / 2;
                const int o = tile * DR + 4 * rq;
                float *dst = (entry == kSharedEntry)
                                 ? p.ws.ysbuf + (size_t)col * H + o
                                 : p.ws.ybuf + ((size_t)col * k + (live ? sm.uni.uslot[entry][col] : 0)) * H + o;
                const int off = partial_index(col, 4 * rq);
                ring_wait(&sm.red_full[rb], (ui / kRed) & 1, abort, hdr, 0x200000u + (uint32_t)ui);
                float4 a[4][4];
#pragma unroll
                for (int t = 0; t < 4; ++t)
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int w = min((t / tpg) * nch + min(c, nch - 1), kConsumerWarps - 1);
                        a[t][c] = *reinterpret_cast<const float4 *>(&sm.red[rb][w][(t % tpg) * 128 + off]);
                    }
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.red_empty[rb]);
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    float4 v = a[t][0];
#pragma unroll
                    for (int c = 1; c < 4; ++c) {
                        const bool on = c < nch;
                        v.x += on ? a[t][c].x : 0.f;
                        v.y += on ? a[t][c].y : 0.f;
                        v.z += on ? a[t][c].z : 0.f;
                        v.w += on ? a[t][c].w : 0.f;
                    }
                    if (live && !*abort)
                        *reinterpret_cast<float4 *>(dst + t * kTileRows) =
                            make_float4(v.x * s2, v.y * s2, v.z * s2, v.w * s2);
                }
                continue;
            }
            if (split) {
                // tile `half` from warps 4 * half .. + 3 (chunk groups 0..3)
                const int o = tile * kOutTile + half * kTileRows + r0;
                float *dst = (entry == kSharedEntry)
                                 ? p.ws.ysbuf + (size_t)col * H + o
                                 : p.ws.ybuf + ((size_t)col * k + (live ? sm.uni.uslot[entry][col] : 0)) * H + o;
                const int off0 = partial_index(col, r0), off1 = partial_index(col, r0 + 4);
                ring_wait(&sm.red_full[rb], (ui / kRed) & 1, abort, hdr, 0x200000u + (uint32_t)ui);
                float4 a[4], c[4];
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    a[w] = *reinterpret_cast<const float4 *>(&sm.red[rb][4 * half + w][off0]);
                    c[w] = *reinterpret_cast<const float4 *>(&sm.red[rb][4 * half + w][off1]);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.red_empty[rb]);
                float4 u = a[0], v = c[0];
#pragma unroll
                for (int w = 1; w < 4; ++w) {
                    u.x += a[w].x; u.y += a[w].y; u.z += a[w].z; u.w += a[w].w;
                    v.x += c[w].x; v.y += c[w].y; v.z += c[w].z; v.w += c[w].w;
                }
                if (live && !*abort) {
                    *reinterpret_cast<float4 *>(dst) = make_float4(u.x * s2, u.y * s2, u.z * s2, u.w * s2);
                    *reinterpret_cast<float4 *>(dst + 4) =
                        make_float4(v.x * s2, v.y * s2, v.z * s2, v.w * s2);
                }
                continue;
            }
            const int nwd = min(kConsumerWarps, K / kChunk);   // warps holding down partials
            const int o = tile * kOutTile + half * kTileRows + r0;
            float *dst = (entry == kSharedEntry)
                             ? p.ws.ysbuf + (size_t)col * H + o
                             : p.ws.ybuf + ((size_t)col * k + (live ? sm.uni.uslot[entry][col] : 0)) * H + o;
            const int off0 = half * 128 + partial_index(col, r0);
            const int off1 = half * 128 + partial_index(col, r0 + 4);
            MOE_TIC(t_ew);
            ring_wait(&sm.red_full[rb], (ui / kRed) & 1, abort, hdr, 0x200000u + (uint32_t)ui);
            MOE_TOC(lane == 0, 27, t_ew);
            MOE_TIC(t_ex);
            float4 a[kConsumerWarps], c[kConsumerWarps];
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                a[w] = *reinterpret_cast<const float4 *>(&sm.red[rb][w][off0]);
                c[w] = *reinterpret_cast<const float4 *>(&sm.red[rb][w][off1]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.red_empty[rb]);
            float ys[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                const bool on = w < nwd;
                ys[0] += on ? a[w].x : 0.f; ys[1] += on ? a[w].y : 0.f;
                ys[2] += on ? a[w].z : 0.f; ys[3] += on ? a[w].w : 0.f;
                ys[4] += on ? c[w].x : 0.f; ys[5] += on ? c[w].y : 0.f;
                ys[6] += on ? c[w].z : 0.f; ys[7] += on ? c[w].w : 0.f;
            }
            if (live && !*abort) {
                *reinterpret_cast<float4 *>(dst) =
                    make_float4(ys[0] * s2, ys[1] * s2, ys[2] * s2, ys[3] * s2);
                *reinterpret_cast<float4 *>(dst + 4) =
                    make_float4(ys[4] * s2, ys[5] * s2, ys[6] * s2, ys[7] * s2);
            }
            MOE_TOC(lane == 0, 28, t_ex);
        }
        named_bar(5, kEpiWarps * 32);
        MOE_PHASE_MARK(lane == 0 && epi_idx == 0, 15);
        if (lane == 0 && epi_idx == 0) grid_arrive_wait(sm.bar, G, abort, hdr, 3u);
        named_bar(5, kEpiWarps * 32);   // both epilogue warps read y in the blend
        asm volatile("bar.arrive 3, %0;" ::"r"(kComputeAndEpi) : "memory");
    } else {
        // ---------------- compute warps ----------------
        const int g = lane >> 2, q = lane & 3;
        int ci = 0;          // slots consumed
        int rs = 0;          // ring slot of the next tile, and its phase parity
        uint32_t rp = 0u;
        auto next_slot = [&]() {
            if (++rs == S) {
                rs = 0;
                rp ^= 1u;
            }
        };
        int ui = 0;   // units handed to the epilogue warps
        // wait until the epilogue warp has consumed the buffer this unit reuses
        auto claim_red = [&]() -> int {
            const int rb = ui % kRed;
            MOE_TIC(t_rw);
            if (ui >= kRed)
                ring_wait(&sm.red_empty[rb], ((ui / kRed) - 1) & 1, abort, hdr,
                          0x300000u + (uint32_t)ui);
            MOE_TOC(tid == 0, 20, t_rw);
            return rb;
        };

        // t layout: compute thread tid owns outputs 8 tid + 2048 g .. + 7
        // (g < NG) and keeps this CTA's partial sums of them.  A unit's down
        // block (its third slot) is applied after the next unit's MMAs, once
        // the epilogue warp has handed over the unit's h: each output's 16
        // products are summed in f16 in two halves of 8 (h scaled so that
        // its largest magnitude lies in [2^8, 2^9): no partial can exceed
        // 8 * 6 * 2^9 < 65504), the halves and the block scale in fp32.
        constexpr int NG = TL ? (MC_GU + 1) / 2 : 1;
        float yacc[NG][8];
#pragma unroll
        for (int gi = 0; gi < NG; ++gi)
#pragma unroll
            for (int i = 0; i < 8; ++i) yacc[gi][i] = 0.f;
        auto tl_apply = [&](int j, int uij, int s, uint32_t par) {
            const int hb = uij % kEpiWarps;
            ring_wait(&sm.h_full[hb], (uij / kEpiWarps) & 1, abort, hdr, 0x600000u + (uint32_t)uij);
            float hv[kTileRows];
#pragma unroll
            for (int i = 0; i < kTileRows; ++i) hv[i] = sm.hsm[hb][i];
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.h_empty[hb]);
            const bool okd = ring_wait(&full[s], par, abort, hdr, 0x700000u + (uint32_t)uij);
            bool live = true;
            float coef;
            if (j < St) {
                coef = sm.gate_val[0] * p.sh_down.scale2;
            } else {
                const int e = (j - St) / It;
                live = sm.ptrs[e].expert >= 0;
                coef = live ? sm.wts[sm.uni.uslot[e][0]] * sm.ptrs[e].scale2[2] : 0.f;
            }
            if (okd && live) {
                float mx = 0.f;
#pragma unroll
                for (int i = 0; i < kTileRows; ++i) mx = fmaxf(mx, fabsf(hv[i]));
                const int ex = max(f16_block_exponent(mx) - 6, -126);
                const float up = exp2i(ex);
                coef *= exp2i(-ex);
                uint32_t h2[kTileRows];
#pragma unroll
                for (int i = 0; i < kTileRows; ++i) h2[i] = pack_f16x2(hv[i] * up, hv[i] * up);
                const uint8_t *blk = ring + (size_t)s * p.slot_bytes;
#pragma unroll
                for (int gi = 0; gi < NG; ++gi) {
                    const int o0 = 8 * tid + 2048 * gi;
                    if (o0 < H) {
                        __half2 acc[2][4];
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                            for (int i = 0; i < 4; ++i) acc[hh][i] = __float2half2_rn(0.f);
#pragma unroll
                        for (int kk = 0; kk < kTileRows; ++kk) {
                            const uint32_t w =
                                *reinterpret_cast<const uint32_t *>(blk + kk * (H / 2) + o0 / 2);
                            uint32_t qv[4];
                            e2m1x8_to_f16x2(w, qv);
                            const __half2 hk = *reinterpret_cast<const __half2 *>(&h2[kk]);
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                acc[kk >> 3][i] = __hfma2(*reinterpret_cast<const __half2 *>(&qv[i]),
                                                          hk, acc[kk >> 3][i]);
                        }
                        const uint2 sc8 = *reinterpret_cast<const uint2 *>(blk + dt_pk + o0);
                        const uint32_t sw[4] = {e4m3x2_to_f16x2(sc8.x & 0xFFFFu),
                                                e4m3x2_to_f16x2(sc8.x >> 16),
                                                e4m3x2_to_f16x2(sc8.y & 0xFFFFu),
                                                e4m3x2_to_f16x2(sc8.y >> 16)};
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float2 sv = __half22float2(*reinterpret_cast<const __half2 *>(&sw[i]));
                            const float2 lo = __half22float2(acc[0][i]);
                            const float2 hi = __half22float2(acc[1][i]);
                            yacc[gi][2 * i] = fmaf(coef * sv.x, lo.x + hi.x, yacc[gi][2 * i]);
                            yacc[gi][2 * i + 1] = fmaf(coef * sv.y, lo.y + hi.y, yacc[gi][2 * i + 1]);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        };
        int tl_j = -1, tl_ui = 0, tl_s = 0;   // the unit whose down block waits
        uint32_t tl_p = 0u;

        // phase C: gate + up (both slots of a unit, the two matrices interleaved)
        {
            uint32_t bx[MC_GU][8][2];
            float inv0, inv1;
            load_b<MC_GU, GV, FMT == 2>(p.x, (size_t)H, allrows, H / kChunk, warp,
                                        kConsumerWarps, lane, bx, inv0, inv1);
            MOE_PHASE_MARK(tid == 0, 5);
            named_bar(4, kLayerThreads);
            sweep_layout();
            const int nch = H / kChunk;
            for (int j = b; j < Tgu; j += G) {
                const int s0 = rs;
                const uint32_t p0 = rp;
                next_slot();
                const int s1 = rs;
                const uint32_t p1 = rp;
                next_slot();
                int s2 = 0;
                uint32_t p2 = 0u;
                if constexpr (TL) {
                    s2 = rs;
                    p2 = rp;
                    next_slot();
                }
                MOE_TIC(t_w);
                const bool ok0 = ring_wait(&full[s0], p0, abort, hdr, (uint32_t)ci);
                bool ok1 = true;
                if constexpr (!kGateFirst) ok1 = ring_wait(&full[s1], p1, abort, hdr, (uint32_t)ci + 1);
                MOE_TOC(tid == 0, 18, t_w);
                MOE_TIC(t_c);
                const uint8_t *sg = ring + (size_t)s0 * p.slot_bytes;
                const uint8_t *su = ring + (size_t)s1 * p.slot_bytes;
                float dg0[4] = {0.f, 0.f, 0.f, 0.f}, dg1[4] = {0.f, 0.f, 0.f, 0.f};
                float du0[4] = {0.f, 0.f, 0.f, 0.f}, du1[4] = {0.f, 0.f, 0.f, 0.f};
                if (FMT == 2 && ghalves == 2) {
                    // K-halves (BF16): this warp's chunks below nh from the
                    // first pair of slots, the rest from the second pair, in
                    // the same chunk order as a whole tile
                    const int nh = nch / 2;
                    const uint32_t hrow = fmt_row_bytes<FMT>(H) / 2;
                    if (ok0 && ok1) {
#pragma unroll
                        for (int m = 0; m < MC_GU; ++m) {
                            const int c = warp + kConsumerWarps * m;
                            if (c < nh) {
                                chunk_mma_t<FMT>(sg, sg, hrow, 0, c, g, q, bx[m], dg0, dg1);
                                chunk_mma_t<FMT>(su, su, hrow, 0, c, g, q, bx[m], du0, du1);
                            }
                        }
                    }
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&empty[s0]);
                        mbar_arrive(&empty[s1]);
                    }
                    const int s2h = rs;
                    const uint32_t p2h = rp;
                    next_slot();
                    const int s3h = rs;
                    const uint32_t p3h = rp;
                    next_slot();
                    const bool ok2 = ring_wait(&full[s2h], p2h, abort, hdr, (uint32_t)ci + 2);
                    const bool ok3 = ring_wait(&full[s3h], p3h, abort, hdr, (uint32_t)ci + 3);
                    const uint8_t *sg2 = ring + (size_t)s2h * p.slot_bytes;
                    const uint8_t *su2 = ring + (size_t)s3h * p.slot_bytes;
                    if (ok2 && ok3) {
#pragma unroll
                        for (int m = 0; m < MC_GU; ++m) {
                            const int c = warp + kConsumerWarps * m;
                            if (c >= nh && c < nch) {
                                chunk_mma_t<FMT>(sg2, sg2, hrow, 0, c - nh, g, q, bx[m], dg0, dg1);
                                chunk_mma_t<FMT>(su2, su2, hrow, 0, c - nh, g, q, bx[m], du0, du1);
                            }
                        }
                    }
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&empty[s2h]);
                        mbar_arrive(&empty[s3h]);
                    }
                    ci += 2;
                } else if constexpr (kGateFirst) {
                    // the gate chunks first; the gate slot goes back to the
                    // producer before the up slot is waited for
                    if (ok0) {
#pragma unroll
                        for (int m = 0; m < MC_GU; ++m) {
                            const int c = warp + kConsumerWarps * m;
                            if (c < nch) {
                                if constexpr (GV) {
                                    float ga, gb;
                                    chunk_gemv(sg, sg + gu_pk, H / 2, H / 16, c, g, q, bx[m], ga, gb);
                                    dg0[0] += ga;
                                    dg0[2] += gb;
                                } else {
                                    chunk_mma_t<FMT>(sg, sg + gu_pk, fmt_row_bytes<FMT>(H),
                                                     fmt_scale_row_bytes<FMT>(H), c, g, q, bx[m], dg0, dg1);
                                }
                            }
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[s0]);
                    ok1 = ring_wait(&full[s1], p1, abort, hdr, (uint32_t)ci + 1);
                    if (ok1) {
#pragma unroll
                        for (int m = 0; m < MC_GU; ++m) {
                            const int c = warp + kConsumerWarps * m;
                            if (c < nch) {
                                if constexpr (GV) {
                                    float ua, ub;
                                    chunk_gemv(su, su + gu_pk, H / 2, H / 16, c, g, q, bx[m], ua, ub);
                                    du0[0] += ua;
                                    du0[2] += ub;
                                } else {
                                    chunk_mma_t<FMT>(su, su + gu_pk, fmt_row_bytes<FMT>(H),
                                                     fmt_scale_row_bytes<FMT>(H), c, g, q, bx[m], du0, du1);
                                }
                            }
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[s1]);
                } else if (ok0 && ok1) {
#pragma unroll
                    for (int m = 0; m < MC_GU; ++m) {
                        const int c = warp + kConsumerWarps * m;
                        if (c < nch) {
                            if constexpr (GV) {
                                float ga, gb, ua, ub;
                                chunk_gemv(sg, sg + gu_pk, H / 2, H / 16, c, g, q, bx[m], ga, gb);
                                chunk_gemv(su, su + gu_pk, H / 2, H / 16, c, g, q, bx[m], ua, ub);
                                dg0[0] += ga;
                                dg0[2] += gb;
                                du0[0] += ua;
                                du0[2] += ub;
                            } else {
                                chunk_mma_t<FMT>(sg, sg + gu_pk, fmt_row_bytes<FMT>(H),
                                                 fmt_scale_row_bytes<FMT>(H), c, g, q, bx[m], dg0, dg1);
                                chunk_mma_t<FMT>(su, su + gu_pk, fmt_row_bytes<FMT>(H),
                                                 fmt_scale_row_bytes<FMT>(H), c, g, q, bx[m], du0, du1);
                            }
                        }
                    }
                }
                if (!(FMT == 2 && ghalves == 2) && !kGateFirst) {
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&empty[s0]);
                        mbar_arrive(&empty[s1]);
                    }
                }
                ci += 2;
                float dg[4], du[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    dg[i] = dg0[i] + dg1[i];
                    du[i] = du0[i] + du1[i];
                }
                MOE_TOC(tid == 0, 19, t_c);
                const int rb = claim_red();
                store_partial(sm.red[rb][warp], dg, g, q, inv0, inv1);
                store_partial(sm.red[rb][warp] + 128, du, g, q, inv0, inv1);
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.red_full[rb]);
                ++ui;
                if constexpr (TL) {
                    if (tl_j >= 0) tl_apply(tl_j, tl_ui, tl_s, tl_p);
                    tl_j = j;
                    tl_ui = ui - 1;
                    tl_s = s2;
                    tl_p = p2;
                }
            }
        }
        MOE_PHASE_MARK(tid == 0, 6);
        if constexpr (TL) {
            if (tl_j >= 0) tl_apply(tl_j, tl_ui, tl_s, tl_p);
            // this CTA's partial outputs; after the grid barrier (taken by
            // the epilogue warp) CTA b sums its slice of outputs over every
            // CTA's partials: tpo threads per output, each adding the CTAs
            // pg, pg + tpo, ... in order, then a fixed butterfly, so the
            // bytes do not depend on timing
            float *ypart = p.ws.ypart + (size_t)b * H;
#pragma unroll
            for (int gi = 0; gi < NG; ++gi) {
                const int o0 = 8 * tid + 2048 * gi;
                if (o0 < H) {
                    *reinterpret_cast<float4 *>(ypart + o0) =
                        make_float4(yacc[gi][0], yacc[gi][1], yacc[gi][2], yacc[gi][3]);
                    *reinterpret_cast<float4 *>(ypart + o0 + 4) =
                        make_float4(yacc[gi][4], yacc[gi][5], yacc[gi][6], yacc[gi][7]);
                }
            }
            named_bar(3, kComputeAndEpi);   // every partial of this CTA stored
            named_bar(3, kComputeAndEpi);   // the grid barrier passed
            MOE_PHASE_MARK(tid == 0, 7);
            const int per = (H + G - 1) / G;
            int lg = 4;
            while (lg > 0 && (per << lg) > kConsumerWarps * 32) --lg;
            const int tpo = 1 << lg;
            const int oi = tid >> lg, pg = tid & (tpo - 1);
            const int o = b * per + oi;
            const bool mine = oi < per && o < H;
            const float *src = p.ws.ypart + (mine ? o : 0);
            float s = 0.f;
            for (int b0 = pg; b0 < G; b0 += 8 * tpo) {
                float v[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) v[i] = ld_cg(src + (size_t)min(b0 + tpo * i, G - 1) * H);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (b0 + tpo * i < G) s += v[i];
            }
            for (int off = tpo >> 1; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
            if (mine && pg == 0 && !*abort) p.out[o] = f2bf16_rn(s);
            MOE_PHASE_MARK(tid == 0, 9);
            return;
        }
        // wait until the epilogue warp has passed the grid barrier (every h written)
        named_bar(2, kComputeAndEpi);
        MOE_PHASE_MARK(tid == 0, 7);

        // phase D: down, 32 output rows per unit (two MMA tiles, four chains).
        // The units of one entry run in an inner loop that only waits,
        // multiplies and hands the partial sums over; the entry's h
        // fragments are loaded once before it.
        {
            uint32_t bh[MC_D][8][2];
            float inv0 = 1.f, inv1 = 1.f;
            int j = d_begin;
            while (j < d_end) {
                int entry, K, jend;
                uint32_t mask;
                if (j < Sd) {
                    entry = kSharedEntry;
                    K = p.Is;
                    mask = allrows;
                    jend = min(Sd, d_end);
                } else {
                    entry = (j - Sd) / Hd;
                    K = p.I;
                    mask = sm.uni.rowmask[entry];
                    jend = min(Sd + (entry + 1) * Hd, d_end);
                }
                const int nch = K / kChunk;
                const uint32_t rowb = fmt_row_bytes<FMT>(K), scb = fmt_scale_row_bytes<FMT>(K);
                // wide units: this warp's chunk and tile group
                // (split units: chunk group warp % 4, tile warp / 4)
                const int cw = wide ? warp % nch : (split ? warp % 4 : warp);
                const int gw = wide ? warp / nch : (split ? warp / 4 : 0);
                const int tpg = nch / 2;
                MOE_TIC(t_b);
                load_b<MC_D, GV, FMT == 2>(p.ws.hbuf + (size_t)entry * kMaxRows * p.ws.inter_max,
                             (size_t)p.ws.inter_max, mask, nch, cw,
                             wide ? nch : (split ? 4 : kConsumerWarps), lane, bh, inv0, inv1);
                MOE_TOC(tid == 0, 21, t_b);
                for (; j < jend; ++j) {
                    if constexpr (kDownParts) {
                        // FP8 / BF16 down unit in K-parts of down_pc chunks,
                        // one slot each (DR row segments): this warp's chunks
                        // in the same order as from a whole tile
                        if (nch > p.down_pc) {
                            float a0[4] = {0.f, 0.f, 0.f, 0.f}, a1[4] = {0.f, 0.f, 0.f, 0.f};
                            float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
                            for (int k0 = 0; k0 < nch; k0 += p.down_pc) {
                                const int nc = min(p.down_pc, nch - k0);
                                const int segb = (int)fmt_row_bytes<FMT>(nc * kChunk);
                                const int s = rs;
                                const uint32_t par = rp;
                                next_slot();
                                const bool ok = ring_wait(&full[s], par, abort, hdr, (uint32_t)ci);
                                const uint8_t *st = ring + (size_t)s * p.slot_bytes;
                                if (ok) {
#pragma unroll
                                    for (int m = 0; m < MC_D; ++m) {
                                        const int c = split ? cw + 4 * m : warp + kConsumerWarps * m;
                                        if (c < k0 || c >= k0 + nc) continue;
                                        if (split) {
                                            chunk_mma_t<FMT>(st + gw * kTileRows * segb, st, segb, 0,
                                                             c - k0, g, q, bh[m], a0, a1);
                                        } else {
                                            chunk_mma_t<FMT>(st, st, segb, 0, c - k0, g, q, bh[m], a0, a1);
                                            chunk_mma_t<FMT>(st + kTileRows * segb, st, segb, 0, c - k0, g,
                                                             q, bh[m], c0, c1);
                                        }
                                    }
                                }
                                __syncwarp();
                                if (lane == 0) mbar_arrive(&empty[s]);
                                ++ci;
                            }
                            float da[4], dc[4];
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                da[i] = a0[i] + a1[i];
                                dc[i] = c0[i] + c1[i];
                            }
                            const int rb = claim_red();
                            store_partial(sm.red[rb][warp], da, g, q, inv0, inv1);
                            store_partial(sm.red[rb][warp] + 128, dc, g, q, inv0, inv1);
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&sm.red_full[rb]);
                            ++ui;
                            continue;
                        }
                    }
                    const int s = rs;
                    const uint32_t par = rp;
                    next_slot();
                    MOE_TIC(t_dw);
                    const bool ok = ring_wait(&full[s], par, abort, hdr, (uint32_t)ci);
                    MOE_TOC(tid == 0, 22, t_dw);
                    MOE_TIC(t_dc);
                    const uint8_t *st = ring + (size_t)s * p.slot_bytes;
                    const uint8_t *sc = st + DR * rowb;
                    float a0[4] = {0.f, 0.f, 0.f, 0.f}, a1[4] = {0.f, 0.f, 0.f, 0.f};
                    float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
                    if (wide) {
                        // tiles gw * tpg .. + tpg - 1 of the unit at chunk cw
                        const int t0 = gw * tpg, t1 = t0 + (tpg > 1 ? 1 : 0);
                        if (ok) {
                            if constexpr (GV) {
                                float ya, yb, yc, yd;
                                chunk_gemv(st + t0 * kTileRows * rowb, sc + t0 * kTileRows * scb, rowb,
                                           scb, cw, g, q, bh[0], ya, yb);
                                chunk_gemv(st + t1 * kTileRows * rowb, sc + t1 * kTileRows * scb, rowb,
                                           scb, cw, g, q, bh[0], yc, yd);
                                a0[0] = ya;
                                a0[2] = yb;
                                c0[0] = yc;
                                c0[2] = yd;
                            } else {
                                chunk_mma_t<FMT>(st + t0 * kTileRows * rowb, sc + t0 * kTileRows * scb, rowb,
                                          scb, cw, g, q, bh[0], a0, a1);
                                chunk_mma_t<FMT>(st + t1 * kTileRows * rowb, sc + t1 * kTileRows * scb, rowb,
                                          scb, cw, g, q, bh[0], c0, c1);
                            }
                        }
                    } else if (split) {
                        // tile gw of the unit at chunks cw + 4 m
                        if (ok) {
#pragma unroll
                            for (int m = 0; m < MC_D; ++m) {
                                const int c = cw + 4 * m;
                                if (c < nch) {
                                    if constexpr (GV) {
                                        float ya, yb;
                                        chunk_gemv(st + gw * kTileRows * rowb, sc + gw * kTileRows * scb,
                                                   rowb, scb, c, g, q, bh[m], ya, yb);
                                        a0[0] += ya;
                                        a0[2] += yb;
                                    } else {
                                        chunk_mma_t<FMT>(st + gw * kTileRows * rowb, sc + gw * kTileRows * scb,
                                                  rowb, scb, c, g, q, bh[m], a0, a1);
                                    }
                                }
                            }
                        }
                    } else if (ok) {
#pragma unroll
                        for (int m = 0; m < MC_D; ++m) {
                            const int c = warp + kConsumerWarps * m;
                            if (c < nch) {
                                if constexpr (GV) {
                                    float ya, yb, yc, yd;
                                    chunk_gemv(st, sc, rowb, scb, c, g, q, bh[m], ya, yb);
                                    chunk_gemv(st + kTileRows * rowb, sc + kTileRows * scb, rowb,
                                               scb, c, g, q, bh[m], yc, yd);
                                    a0[0] += ya;
                                    a0[2] += yb;
                                    c0[0] += yc;
                                    c0[2] += yd;
                                } else {
                                    chunk_mma_t<FMT>(st, sc, rowb, scb, c, g, q, bh[m], a0, a1);
                                    chunk_mma_t<FMT>(st + kTileRows * rowb, sc + kTileRows * scb, rowb,
                                              scb, c, g, q, bh[m], c0, c1);
                                }
                            }
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[s]);
                    ++ci;
                    float da[4], dc[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        da[i] = a0[i] + a1[i];
                        dc[i] = c0[i] + c1[i];
                    }
                    MOE_TOC(tid == 0, 23, t_dc);
                    const int rb = claim_red();
                    store_partial(sm.red[rb][warp], da, g, q, inv0, inv1);
                    store_partial(sm.red[rb][warp] + 128, dc, g, q, inv0, inv1);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sm.red_full[rb]);
                    ++ui;
                }
            }
        }
        MOE_PHASE_MARK(tid == 0, 8);
        // wait until the epilogue warp has passed the grid barrier (every y written)
        named_bar(3, kComputeAndEpi);
        MOE_PHASE_MARK(tid == 0, 12);
    }

    // ---------------- phase E: blend, spread over the CTAs ----------------
    // Items (32-row output tile, token row) go to the compute and epilogue
    // warps of all CTAs, one warp per item, one output per lane.
    const int items = Ho * p.rows;
    const int bw = warp == kEpiWarp2 ? kConsumerWarps + 1 : warp;   // blend warp index
    for (int it = b + G * bw; it < items; it += G * (kConsumerWarps + kEpiWarps)) {
        const int t = it / p.rows, r = it % p.rows;
        const int o = t * kOutTile + lane;
        const float ysv = ld_cg(p.ws.ysbuf + (size_t)r * H + o);
        float acc = 0.f;
        // slots in order, eight loads in flight at a time
        for (int s0 = 0; s0 < k; s0 += 8) {
            float yv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                yv[i] = ld_cg(p.ws.ybuf + ((size_t)r * k + min(s0 + i, k - 1)) * H + o);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (s0 + i < k) acc = fmaf(sm.wts[r * k + s0 + i], yv[i], acc);
        }
        if (p.has_shared) acc = fmaf(sm.gate_val[r], ysv, acc);
        if (!*abort) p.out[(size_t)r * H + o] = f2bf16_rn(acc);
    }
    MOE_PHASE_MARK(tid == 0, 9);
}

// The sixteen (MC_GU, MC_D) instantiations of one top-k class, projection
// variant and expert format.
template <int TK, bool GV, int FMT = 0>
void *layer_kernel_table(int mc_gu, int mc_d) {
    static void *const tab[4][4] = {
        {(void *)moe_layer_kernel<1, 1, TK, GV, false, FMT>, (void *)moe_layer_kernel<1, 2, TK, GV, false, FMT>,
         (void *)moe_layer_kernel<1, 3, TK, GV, false, FMT>, (void *)moe_layer_kernel<1, 4, TK, GV, false, FMT>},
        {(void *)moe_layer_kernel<2, 1, TK, GV, false, FMT>, (void *)moe_layer_kernel<2, 2, TK, GV, false, FMT>,
         (void *)moe_layer_kernel<2, 3, TK, GV, false, FMT>, (void *)moe_layer_kernel<2, 4, TK, GV, false, FMT>},
        {(void *)moe_layer_kernel<3, 1, TK, GV, false, FMT>, (void *)moe_layer_kernel<3, 2, TK, GV, false, FMT>,
         (void *)moe_layer_kernel<3, 3, TK, GV, false, FMT>, (void *)moe_layer_kernel<3, 4, TK, GV, false, FMT>},
        {(void *)moe_layer_kernel<4, 1, TK, GV, false, FMT>, (void *)moe_layer_kernel<4, 2, TK, GV, false, FMT>,
         (void *)moe_layer_kernel<4, 3, TK, GV, false, FMT>, (void *)moe_layer_kernel<4, 4, TK, GV, false, FMT>}};
    if (mc_gu < 1 || mc_gu > 4 || mc_d < 1 || mc_d > 4) return nullptr;
    return tab[mc_gu - 1][mc_d - 1];
}

// The K-part instantiations of one top-k class and expert format: MC_GU
// 1..4 x MC_D 2..4, those that down_parts_possible allows (null otherwise).
template <int MC_GU, int MC_D, int TK, int FMT>
void *layer_kernel_kp_entry() {
    if constexpr (down_parts_possible(FMT, MC_D))
        return (void *)moe_layer_kernel<MC_GU, MC_D, TK, false, false, FMT, true>;
    else
        return nullptr;
}
template <int TK, int FMT>
void *layer_kernel_kp_table(int mc_gu, int mc_d) {
    static void *const tab[4][3] = {
        {layer_kernel_kp_entry<1, 2, TK, FMT>(), layer_kernel_kp_entry<1, 3, TK, FMT>(),
         layer_kernel_kp_entry<1, 4, TK, FMT>()},
        {layer_kernel_kp_entry<2, 2, TK, FMT>(), layer_kernel_kp_entry<2, 3, TK, FMT>(),
         layer_kernel_kp_entry<2, 4, TK, FMT>()},
        {layer_kernel_kp_entry<3, 2, TK, FMT>(), layer_kernel_kp_entry<3, 3, TK, FMT>(),
         layer_kernel_kp_entry<3, 4, TK, FMT>()},
        {layer_kernel_kp_entry<4, 2, TK, FMT>(), layer_kernel_kp_entry<4, 3, TK, FMT>(),
         layer_kernel_kp_entry<4, 4, TK, FMT>()}};
    if (mc_gu < 1 || mc_gu > 4 || mc_d < 2 || mc_d > 4) return nullptr;
    return tab[mc_gu - 1][mc_d - 2];
}

// The t-layout (fused one-row) instantiations of one top-k class: MC_GU
// 1..4, both projection variants.
template <int TK>
void *layer_kernel_t_table(int mc_gu, bool gv) {
    static void *const tab[2][4] = {
        {(void *)moe_layer_kernel<1, 1, TK, false, true>, (void *)moe_layer_kernel<2, 1, TK, false, true>,
         (void *)moe_layer_kernel<3, 1, TK, false, true>, (void *)moe_layer_kernel<4, 1, TK, false, true>},
        {(void *)moe_layer_kernel<1, 1, TK, true, true>, (void *)moe_layer_kernel<2, 1, TK, true, true>,
         (void *)moe_layer_kernel<3, 1, TK, true, true>, (void *)moe_layer_kernel<4, 1, TK, true, true>}};
    if (mc_gu < 1 || mc_gu > 4) return nullptr;
    return tab[gv ? 1 : 0][mc_gu - 1];
}

}  // namespace moe
