// moe_expert.cu -- the NVFP4 (W4A16) expert sweep: gate+up with SiLU*up, then
// down with the routing-weighted sum and the shared-expert blend.
//
// Each union expert's weights are streamed from HBM once for all the token
// rows that selected it (page "Function forward_moe", RETRACTED note:
// w4a16_gemv_sw_moe_batchm_mR sweeps each union expert once); the shared
// expert is one more entry whose row mask holds every row (the shared-expert
// note: same weights for every row, run once over all of them).  The math of
// each entry is that of forward_token_major.rs
// (moe_expert_gate_up_shared_prefill, moe_expert_silu_down_shared_prefill,
// moe_weighted_sum_blend_prefill).
//
// Work unit: one 16-row tile of an entry's matrix (gate and up together in
// the first kernel).  The tile is contiguous in the [N][K/2] layout, so one
// producer thread stages it in shared memory with bulk (TMA) copies behind an
// mbarrier ring; the consumer warps split K into fixed 128-input chunks
// (chunk c -> warp c mod W), unpack E2M1 x E4M3 to f16 in registers (exact),
// and multiply on the tensor cores (mma.sync m16n8k16, f16 in, fp32
// accumulate) against the token rows as the 8 MMA columns.
//
// The token rows enter the MMA as f16 after a power-of-two scale chosen per
// (warp, row) from the largest magnitude in that warp's chunks; the scale is
// undone in fp32 after the MMAs.  bf16 -> f16 is exact for every value within
// 2^-28 of that largest magnitude.
//
// Determinism: the result for (entry expert e, row r) depends only on e's
// weights and row r's inputs -- MMA columns are independent, the K split is
// fixed by K alone, the cross-warp sum runs in warp order, and the weighted
// sum runs in slot order -- so the union sweep and the per-row mode (every
// (row, slot) pair its own entry) produce the same bytes.
#include <cuda_runtime.h>

#include "moe_device.cuh"

namespace moe {

// ---------------------------------------------------------------------------
// Shared pieces
// ---------------------------------------------------------------------------

struct Ring {
    uint64_t *full;
    uint64_t *empty;
    volatile int *abort;
};

// Wait on a ring barrier; gives up (and makes every later wait give up) once
// the CTA's abort flag is set or the wait exceeds its bound.
__device__ __forceinline__ bool ring_wait(const Ring &rg, uint64_t *bar, uint32_t parity,
                                          WsHeader *hdr, uint32_t info) {
    if (*rg.abort) return false;
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (*rg.abort) return false;
        if (clock64() - t0 > kWaitLimitCycles) {
            *rg.abort = 1;
            record_fault(hdr, MOE_DEV_WAIT_TIMEOUT, info);
            return false;
        }
    }
    return true;
}

// One 128-input chunk of a 16-row tile against the B fragments of that
// chunk.  Lane (g = lane/4, q = lane%4) reads 16 bytes (32 inputs) of rows g
// and g+8 at input offset q*32 inside the chunk, plus their two E4M3 scales.
// MMA step s (0..7) uses inputs 4s..4s+3 of that 32-input slice: logical k
// (2q, 2q+1) <- inputs (4s, 4s+1) and (2q+8, 2q+9) <- (4s+2, 4s+3); the B
// fragments hold the token rows at the same inputs.
__device__ __forceinline__ void chunk_mma(const uint8_t *pk, const uint8_t *sc, int row_bytes,
                                          int sc_row_bytes, int c, int g, int q,
                                          const uint32_t (&b)[8][2], float (&d)[4]) {
    const uint4 wa = *reinterpret_cast<const uint4 *>(pk + g * row_bytes + c * 64 + q * 16);
    const uint4 wb =
        *reinterpret_cast<const uint4 *>(pk + (g + 8) * row_bytes + c * 64 + q * 16);
    const uint32_t sa = *reinterpret_cast<const uint16_t *>(sc + g * sc_row_bytes + c * 8 + q * 2);
    const uint32_t sb =
        *reinterpret_cast<const uint16_t *>(sc + (g + 8) * sc_row_bytes + c * 8 + q * 2);
    const uint32_t fa = e4m3x2_to_f16x2(sa), fb = e4m3x2_to_f16x2(sb);
    const uint32_t sa0 = bcast_lo(fa), sa1 = bcast_hi(fa);
    const uint32_t sb0 = bcast_lo(fb), sb1 = bcast_hi(fb);
    const uint32_t wA[4] = {wa.x, wa.y, wa.z, wa.w};
    const uint32_t wB[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        uint32_t ha[4], hb[4];
        e2m1x8_to_f16x2(wA[t], ha);
        e2m1x8_to_f16x2(wB[t], hb);
        const uint32_t scA = t < 2 ? sa0 : sa1;
        const uint32_t scB = t < 2 ? sb0 : sb1;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            ha[i] = hmul2(ha[i], scA);
            hb[i] = hmul2(hb[i], scB);
        }
        mma_f16_16816(d, ha[0], hb[0], ha[1], hb[1], b[2 * t][0], b[2 * t][1]);
        mma_f16_16816(d, ha[2], hb[2], ha[3], hb[3], b[2 * t + 1][0], b[2 * t + 1][1]);
    }
}

// Load the B fragments of one token-row matrix (x or h) for this warp's
// chunks: lane (n = lane/4, q = lane%4) takes row n's 32 inputs at offset
// c*128 + q*32.  Rows not in `mask` become zero.  Returns the per-column
// unscale factors 2^-e for the D columns 2q and 2q+1 in inv0 / inv1.
template <int MAXC>
__device__ __forceinline__ void load_b(const uint16_t *rows_base, size_t row_stride,
                                       uint32_t mask, int nchunk, int warp, int nwarps,
                                       int lane, uint32_t (&b)[MAXC][8][2], float &inv0,
                                       float &inv1) {
    const int n = lane >> 2, q = lane & 3;
    const bool on = (mask >> n) & 1u;
    float mx = 0.f;
#pragma unroll
    for (int m = 0; m < MAXC; ++m) {
        const int c = warp + nwarps * m;
        if (on && c < nchunk) {
            const uint16_t *src = rows_base + (size_t)n * row_stride + c * kChunk + q * 32;
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const uint4 xv = ld_cg_v4(src + 8 * v);
                const uint32_t w[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                for (int t = 0; t < 4; ++t)
                    mx = fmaxf(mx, fmaxf(fabsf(bf16_lo(w[t])), fabsf(bf16_hi(w[t]))));
            }
        }
    }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const int e = f16_block_exponent(mx);
    const float up = exp2i(e);
#pragma unroll
    for (int m = 0; m < MAXC; ++m) {
        const int c = warp + nwarps * m;
        if (on && c < nchunk) {
            const uint16_t *src = rows_base + (size_t)n * row_stride + c * kChunk + q * 32;
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const uint4 xv = ld_cg_v4(src + 8 * v);
                // inputs 8v..8v+7 -> steps 2v (4 inputs) and 2v+1
                b[m][2 * v][0] = pack_f16x2(bf16_lo(xv.x) * up, bf16_hi(xv.x) * up);
                b[m][2 * v][1] = pack_f16x2(bf16_lo(xv.y) * up, bf16_hi(xv.y) * up);
                b[m][2 * v + 1][0] = pack_f16x2(bf16_lo(xv.z) * up, bf16_hi(xv.z) * up);
                b[m][2 * v + 1][1] = pack_f16x2(bf16_lo(xv.w) * up, bf16_hi(xv.w) * up);
            }
        } else {
#pragma unroll
            for (int s = 0; s < 8; ++s) b[m][s][0] = b[m][s][1] = 0u;
        }
    }
    const float inv = exp2i(-e);
    inv0 = __shfl_sync(0xffffffffu, inv, 8 * q);
    inv1 = __shfl_sync(0xffffffffu, inv, 8 * q + 4);
}

// D fragment (lane g, q: rows g / g+8, columns 2q / 2q+1) -> smem [16][8].
__device__ __forceinline__ void store_partial(float *dst, const float (&d)[4], int g, int q,
                                              float inv0, float inv1) {
    dst[g * 8 + 2 * q] = d[0] * inv0;
    dst[g * 8 + 2 * q + 1] = d[1] * inv1;
    dst[(g + 8) * 8 + 2 * q] = d[2] * inv0;
    dst[(g + 8) * 8 + 2 * q + 1] = d[3] * inv1;
}

// ---------------------------------------------------------------------------
// Gate + up + SiLU*up
// ---------------------------------------------------------------------------
//
// Units: the shared expert's Is/16 tiles first, then U * I/16 union tiles
// (entry-major); CTA b takes units b, b + G, b + 2G, ...  The shared units
// need no routing, so the producer stages them before waiting for the route
// kernel.  Output: h[entry][row][i] = bf16(silu(g) * v).

template <int MAXC>
__global__ void __launch_bounds__((kConsumerWarps + 1) * 32, 1)
    moe_gate_up_kernel(const ExpertParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int s_abort;

    const int H = p.H, S = p.stages;
    const uint32_t pk_bytes = kTileRows * H / 2;
    const uint32_t sc_bytes = kTileRows * H / 16;
    float *red = reinterpret_cast<float *>(smem + (size_t)S * p.stage_bytes);
    uint64_t *full = reinterpret_cast<uint64_t *>(red + 2 * kConsumerWarps * 256);
    uint64_t *empty = full + S;
    Ring rg{full, empty, &s_abort};

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        fence_mbar_init();
        s_abort = 0;
    }
    __syncthreads();
    pdl_trigger();

    const int It = p.I / kTileRows;
    const int St = p.has_shared ? p.Is / kTileRows : 0;
    const int G = gridDim.x;
    WsHeader *hdr = p.ws.hdr;

    if (warp == kConsumerWarps) {
        // ---------------- producer ----------------
        if (lane == 0) {
            const uint64_t pol = l2_evict_first_policy();
            int T = -1;
            for (int i = 0, j = blockIdx.x;; ++i, j += G) {
                if (j >= St && T < 0) {
                    pdl_wait();
                    T = St + ld_cg(&p.ws.uni->num_union) * It;
                }
                if (T >= 0 && j >= T) break;
                const int s = i % S;
                if (i >= S && !ring_wait(rg, &empty[s], ((i / S) - 1) & 1, hdr, (uint32_t)j))
                    break;
                const uint8_t *gp, *gs, *upk, *us;
                if (j < St) {
                    gp = p.sh_gate.packed + (size_t)j * pk_bytes;
                    gs = p.sh_gate.scales + (size_t)j * sc_bytes;
                    upk = p.sh_up.packed + (size_t)j * pk_bytes;
                    us = p.sh_up.scales + (size_t)j * sc_bytes;
                } else {
                    const int u = (j - St) / It, tile = (j - St) % It;
                    const PtrEntry *e = p.ws.ptrs + u;
                    if (ld_cg(&e->expert) < 0) {
                        mbar_arrive(&full[s]);
                        continue;
                    }
                    gp = ld_cg(&e->packed[0]) + (size_t)tile * pk_bytes;
                    gs = ld_cg(&e->scales[0]) + (size_t)tile * sc_bytes;
                    upk = ld_cg(&e->packed[1]) + (size_t)tile * pk_bytes;
                    us = ld_cg(&e->scales[1]) + (size_t)tile * sc_bytes;
                }
                uint8_t *st = smem + (size_t)s * p.stage_bytes;
                mbar_arrive_expect_tx(&full[s], 2 * (pk_bytes + sc_bytes));
                bulk_g2s(st, gp, pk_bytes, &full[s], pol);
                bulk_g2s(st + pk_bytes, gs, sc_bytes, &full[s], pol);
                bulk_g2s(st + pk_bytes + sc_bytes, upk, pk_bytes, &full[s], pol);
                bulk_g2s(st + 2 * pk_bytes + sc_bytes, us, sc_bytes, &full[s], pol);
            }
        }
        return;
    }

    // ---------------- consumers ----------------
    pdl_wait();
    const int U = ld_cg(&p.ws.uni->num_union);
    const int T = St + U * It;
    const int g = lane >> 2, q = lane & 3;
    const int nchunk = H / kChunk;
    const uint32_t allrows = (1u << p.rows) - 1u;

    uint32_t b[MAXC][8][2];
    float inv0, inv1;
    load_b<MAXC>(p.x, (size_t)H, allrows, nchunk, warp, kConsumerWarps, lane, b, inv0, inv1);

    const int NT = kConsumerWarps * 32;
    for (int i = 0, j = blockIdx.x; j < T; ++i, j += G) {
        const int s = i % S;
        const bool ok = ring_wait(rg, &full[s], (i / S) & 1, hdr, (uint32_t)j);
        const uint8_t *st = smem + (size_t)s * p.stage_bytes;
        float dg[4] = {0.f, 0.f, 0.f, 0.f}, du[4] = {0.f, 0.f, 0.f, 0.f};
        if (ok) {
#pragma unroll
            for (int m = 0; m < MAXC; ++m) {
                const int c = warp + kConsumerWarps * m;
                if (c < nchunk) {
                    chunk_mma(st, st + pk_bytes, H / 2, H / 16, c, g, q, b[m], dg);
                    chunk_mma(st + pk_bytes + sc_bytes, st + 2 * pk_bytes + sc_bytes, H / 2,
                              H / 16, c, g, q, b[m], du);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);

        float *rb = red + ((i & 1) * kConsumerWarps + warp) * 256;
        store_partial(rb, dg, g, q, inv0, inv1);
        store_partial(rb + 128, du, g, q, inv0, inv1);
        named_bar(1, NT);

        if (threadIdx.x < 128) {
            const int t = threadIdx.x, row = t >> 3, col = t & 7;
            int entry, tile;
            float s2g, s2u;
            uint32_t mask;
            bool valid = !s_abort;
            if (j < St) {
                entry = kSharedEntry;
                tile = j;
                s2g = p.sh_gate.scale2;
                s2u = p.sh_up.scale2;
                mask = allrows;
            } else {
                entry = (j - St) / It;
                tile = (j - St) % It;
                const PtrEntry *e = p.ws.ptrs + entry;
                valid = valid && ld_cg(&e->expert) >= 0;
                s2g = ld_cg(&e->scale2[0]);
                s2u = ld_cg(&e->scale2[1]);
                mask = ld_cg(&p.ws.uni->rowmask[entry]);
            }
            const float *r0 = red + (i & 1) * kConsumerWarps * 256;
            float gs = 0.f, us = 0.f;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                gs += r0[w * 256 + t];
                us += r0[w * 256 + 128 + t];
            }
            if (valid && ((mask >> col) & 1u)) {
                const float gv = gs * s2g, uv = us * s2u;
                const float hv = gv / (1.f + expf(-gv)) * uv;
                p.ws.hbuf[((size_t)entry * kMaxRows + col) * p.ws.inter_max + tile * kTileRows +
                          row] = f2bf16_rn(hv);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Down + routing-weighted sum + shared-expert blend
// ---------------------------------------------------------------------------
//
// Units: the shared expert's H/16 down tiles first, then U * H/16 union tiles
// (entry-major); CTA b takes a contiguous range of units, so consecutive
// units mostly share an entry and its h fragments stay in registers.  Each
// unit writes y (fp32) for the rows of its mask; the CTA that completes the
// last entry of an output tile (a per-tile arrival counter) forms
//   out[r][o] = bf16( sum_{slot < k} w[r][slot] * y[r][slot][o] + g_r * ys[r][o] )
// in slot order and resets the counter.

template <int MAXC>
__global__ void __launch_bounds__((kConsumerWarps + 1) * 32, 1)
    moe_down_kernel(const ExpertParams p, const int W) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int s_abort;
    __shared__ int s_last;

    const int H = p.H, S = p.stages;
    const int Kmax = p.ws.inter_max;
    float *red = reinterpret_cast<float *>(smem + (size_t)S * p.stage_bytes);
    uint64_t *full = reinterpret_cast<uint64_t *>(red + 2 * kConsumerWarps * 128);
    uint64_t *empty = full + S;
    Ring rg{full, empty, &s_abort};

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], W);
        }
        fence_mbar_init();
        s_abort = 0;
    }
    __syncthreads();
    pdl_trigger();
    pdl_wait();

    const int Ht = H / kTileRows;
    const int Sd = p.has_shared ? Ht : 0;
    const int U = ld_cg(&p.ws.uni->num_union);
    const int T = Sd + U * Ht;
    const int G = gridDim.x;
    const int begin = (int)((long long)blockIdx.x * T / G);
    const int end = (int)((long long)(blockIdx.x + 1) * T / G);
    const int n_entries = U + (p.has_shared ? 1 : 0);
    WsHeader *hdr = p.ws.hdr;
    (void)Kmax;

    if (warp == W) {
        // ---------------- producer ----------------
        if (lane == 0) {
            const uint64_t pol = l2_evict_first_policy();
            for (int i = 0, j = begin; j < end; ++i, ++j) {
                const int s = i % S;
                if (i >= S && !ring_wait(rg, &empty[s], ((i / S) - 1) & 1, hdr, (uint32_t)j))
                    break;
                const uint8_t *dp, *ds;
                int K;
                if (j < Sd) {
                    K = p.Is;
                    dp = p.sh_down.packed + (size_t)j * kTileRows * (K / 2);
                    ds = p.sh_down.scales + (size_t)j * kTileRows * (K / 16);
                } else {
                    const int u = (j - Sd) / Ht, tile = (j - Sd) % Ht;
                    const PtrEntry *e = p.ws.ptrs + u;
                    if (ld_cg(&e->expert) < 0) {
                        mbar_arrive(&full[s]);
                        continue;
                    }
                    K = p.I;
                    dp = ld_cg(&e->packed[2]) + (size_t)tile * kTileRows * (K / 2);
                    ds = ld_cg(&e->scales[2]) + (size_t)tile * kTileRows * (K / 16);
                }
                const uint32_t pkb = kTileRows * K / 2, scb = kTileRows * K / 16;
                uint8_t *st = smem + (size_t)s * p.stage_bytes;
                mbar_arrive_expect_tx(&full[s], pkb + scb);
                bulk_g2s(st, dp, pkb, &full[s], pol);
                bulk_g2s(st + pkb, ds, scb, &full[s], pol);
            }
        }
        return;
    }

    // ---------------- consumers ----------------
    const int g = lane >> 2, q = lane & 3;
    const int NT = W * 32;
    uint32_t b[MAXC][8][2];
    float inv0 = 1.f, inv1 = 1.f;
    int cur_entry = -1;

    for (int i = 0, j = begin; j < end; ++i, ++j) {
        int entry, tile, K;
        uint32_t mask;
        float s2;
        bool valid = true;
        if (j < Sd) {
            entry = kSharedEntry;
            tile = j;
            K = p.Is;
            mask = (1u << p.rows) - 1u;
            s2 = p.sh_down.scale2;
        } else {
            entry = (j - Sd) / Ht;
            tile = (j - Sd) % Ht;
            K = p.I;
            mask = ld_cg(&p.ws.uni->rowmask[entry]);
            const PtrEntry *e = p.ws.ptrs + entry;
            valid = ld_cg(&e->expert) >= 0;
            s2 = ld_cg(&e->scale2[2]);
        }
        const int nchunk = K / kChunk;
        if (entry != cur_entry) {
            load_b<MAXC>(p.ws.hbuf + (size_t)entry * kMaxRows * p.ws.inter_max,
                         (size_t)p.ws.inter_max, mask, nchunk, warp, W, lane, b, inv0, inv1);
            cur_entry = entry;
        }
        const int s = i % S;
        const bool ok = ring_wait(rg, &full[s], (i / S) & 1, hdr, (uint32_t)j);
        const uint8_t *st = smem + (size_t)s * p.stage_bytes;
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        if (ok) {
#pragma unroll
            for (int m = 0; m < MAXC; ++m) {
                const int c = warp + W * m;
                if (c < nchunk)
                    chunk_mma(st, st + kTileRows * K / 2, K / 2, K / 16, c, g, q, b[m], d);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);

        float *rb = red + ((i & 1) * kConsumerWarps + warp) * 128;
        store_partial(rb, d, g, q, inv0, inv1);
        named_bar(1, NT);

        const float *r0 = red + (i & 1) * kConsumerWarps * 128;
        valid = valid && !s_abort;
        for (int t = threadIdx.x; t < 128; t += NT) {
            const int row = t >> 3, col = t & 7;
            float ys = 0.f;
            for (int w = 0; w < W; ++w) ys += r0[w * 128 + t];
            if (valid && ((mask >> col) & 1u)) {
                const int o = tile * kTileRows + row;
                const float yv = ys * s2;
                if (entry == kSharedEntry) {
                    p.ws.ysbuf[(size_t)col * H + o] = yv;
                } else {
                    const int slot = ld_cg(&p.ws.uni->uslot[entry][col]);
                    p.ws.ybuf[((size_t)col * p.k + slot) * H + o] = yv;
                }
            }
        }
        __threadfence();
        named_bar(1, NT);
        if (threadIdx.x == 0) {
            const unsigned old = atomicAdd(&p.ws.tile_cnt[tile], 1u);
            s_last = (old == (unsigned)(n_entries - 1));
        }
        named_bar(1, NT);
        if (s_last) {
            __threadfence();
            for (int t = threadIdx.x; t < p.rows * kTileRows; t += NT) {
                const int r = t / kTileRows, o = tile * kTileRows + t % kTileRows;
                float acc = 0.f;
                for (int sl = 0; sl < p.k; ++sl)
                    acc = fmaf(ld_cg(p.ws.wts + r * p.k + sl),
                               ld_cg(p.ws.ybuf + ((size_t)r * p.k + sl) * H + o), acc);
                if (p.has_shared)
                    acc = fmaf(ld_cg(p.ws.gate_val + r), ld_cg(p.ws.ysbuf + (size_t)r * H + o),
                               acc);
                p.out[(size_t)r * H + o] = f2bf16_rn(acc);
            }
            if (threadIdx.x == 0) p.ws.tile_cnt[tile] = 0u;
        }
    }
}

// ---------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------

template <typename K>
static cudaError_t launch_pdl(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              const ExpertParams &p) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, p);
}

template <typename K>
static cudaError_t launch_pdl_w(K kernel, dim3 grid, dim3 block, size_t smem,
                                cudaStream_t stream, const ExpertParams &p, int W) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, p, W);
}

// Shared memory the expert kernels need besides their stage ring.
size_t gate_up_fixed_smem(int stages) {
    return sizeof(float) * 2 * kConsumerWarps * 256 + 2 * sizeof(uint64_t) * stages;
}
size_t down_fixed_smem(int stages) {
    return sizeof(float) * 2 * kConsumerWarps * 128 + 2 * sizeof(uint64_t) * stages;
}

cudaError_t set_expert_smem_limits(int bytes) {
    cudaError_t e;
    void *gu[4] = {(void *)moe_gate_up_kernel<1>, (void *)moe_gate_up_kernel<2>,
                   (void *)moe_gate_up_kernel<3>, (void *)moe_gate_up_kernel<4>};
    void *dn[4] = {(void *)moe_down_kernel<1>, (void *)moe_down_kernel<2>,
                   (void *)moe_down_kernel<3>, (void *)moe_down_kernel<4>};
    for (int i = 0; i < 4; ++i) {
        if ((e = cudaFuncSetAttribute(gu[i], cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      bytes)) != cudaSuccess)
            return e;
        if ((e = cudaFuncSetAttribute(dn[i], cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      bytes)) != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

cudaError_t launch_gate_up(const ExpertParams &p, int grid, size_t smem, int maxc,
                           cudaStream_t stream) {
    const dim3 block((kConsumerWarps + 1) * 32);
    switch (maxc) {
        case 1: return launch_pdl(moe_gate_up_kernel<1>, dim3(grid), block, smem, stream, p);
        case 2: return launch_pdl(moe_gate_up_kernel<2>, dim3(grid), block, smem, stream, p);
        case 3: return launch_pdl(moe_gate_up_kernel<3>, dim3(grid), block, smem, stream, p);
        case 4: return launch_pdl(moe_gate_up_kernel<4>, dim3(grid), block, smem, stream, p);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_down(const ExpertParams &p, int grid, int W, size_t smem, int maxc,
                        cudaStream_t stream) {
    const dim3 block((W + 1) * 32);
    switch (maxc) {
        case 1: return launch_pdl_w(moe_down_kernel<1>, dim3(grid), block, smem, stream, p, W);
        case 2: return launch_pdl_w(moe_down_kernel<2>, dim3(grid), block, smem, stream, p, W);
        case 3: return launch_pdl_w(moe_down_kernel<3>, dim3(grid), block, smem, stream, p, W);
        case 4: return launch_pdl_w(moe_down_kernel<4>, dim3(grid), block, smem, stream, p, W);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace moe
