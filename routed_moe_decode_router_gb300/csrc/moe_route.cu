// moe_route.cu -- router projection, batched top-k and the union of the
// selected experts, all on the device.
//
// Router (forward_ep.rs / forward_token_major.rs: dense_gemv / dense_gemm for
// a bf16 gate, w4a16_decode_gemv / w4a16_gemm for an NVFP4 gate): one warp
// per router row computes the logits of that expert for every token row with
// fp32 accumulation.  The shared-expert gate vector rides along as one more
// row, giving sigmoid(x . shared_expert_gate) per token row.
//
// Top-k (forward_token_major.rs: moe_topk_softmax_batched,
// moe_topk_sigmoid_batched; forward_ep.rs: moe_topk_softmax) runs in the
// block that finishes last (an atomic ticket), one warp per token row:
// selection key descending with ties to the lower expert id; softmax selects
// on the logit, sigmoid scoring on sigmoid(logit) + correction bias.  One
// launch covers a sub-chunk of at most 8 rows; a call of more rows launches
// one per sub-chunk.
//
// Union (page "Function forward_moe", RETRACTED and WIDENED notes): the ids
// of all the call's rows (at most 256) are de-duplicated by pairwise scan in
// blocks of 64 -- a position starts a union entry when no earlier position,
// in its own block or an earlier one, holds the same id -- with no sort and
// no copy to the host.  The kernel writes the call's union table and the
// device pointer table of the union experts (the forward_moe page's
// pointer-table upgrade path) into the workspace, for moe_union and for
// calls of several sub-chunks; the layer kernel builds its own copy of a
// sub-chunk's table in shared memory.
#include <cuda_runtime.h>

#include "moe_blocks.cuh"

namespace moe {

// ---------------------------------------------------------------------------
// Router rows
// ---------------------------------------------------------------------------

// acc[r] += sum_h x[r][h] * w[h] over a bf16 row of H values.
__device__ __forceinline__ void dot_bf16_row(const uint16_t *__restrict__ w,
                                             const uint16_t *__restrict__ x, int H, int rows,
                                             int lane, float (&acc)[kMaxRows]) {
#pragma unroll 4
    for (int h0 = lane * 8; h0 < H; h0 += 256) {
        const uint4 wv = ld_nc_v4(w + h0);
        const float wf[8] = {bf16_lo(wv.x), bf16_hi(wv.x), bf16_lo(wv.y), bf16_hi(wv.y),
                             bf16_lo(wv.z), bf16_hi(wv.z), bf16_lo(wv.w), bf16_hi(wv.w)};
#pragma unroll
        for (int r = 0; r < kMaxRows; ++r) {
            if (r < rows) {
                const uint4 xv = *reinterpret_cast<const uint4 *>(x + (size_t)r * H + h0);
                float a = acc[r];
                a = fmaf(bf16_lo(xv.x), wf[0], a);
                a = fmaf(bf16_hi(xv.x), wf[1], a);
                a = fmaf(bf16_lo(xv.y), wf[2], a);
                a = fmaf(bf16_hi(xv.y), wf[3], a);
                a = fmaf(bf16_lo(xv.z), wf[4], a);
                a = fmaf(bf16_hi(xv.z), wf[5], a);
                a = fmaf(bf16_lo(xv.w), wf[6], a);
                a = fmaf(bf16_hi(xv.w), wf[7], a);
                acc[r] = a;
            }
        }
    }
}

// acc[r] += sum_h x[r][h] * (e2m1 * e4m3) over one NVFP4 row; the caller
// applies scale2.  Each lane takes 32 consecutive inputs per step.
__device__ __forceinline__ void dot_nvfp4_row(const uint8_t *__restrict__ packed,
                                              const uint8_t *__restrict__ scales,
                                              const uint16_t *__restrict__ x, int H, int rows,
                                              int lane, float (&acc)[kMaxRows]) {
    for (int base = lane * 32; base < H; base += 1024) {
        const uint4 pv = ld_nc_v4(packed + base / 2);
        const uint32_t sv = *reinterpret_cast<const uint16_t *>(scales + base / 16);
        const uint32_t s2u = e4m3x2_to_f16x2(sv);
        const __half2 s2 = *reinterpret_cast<const __half2 *>(&s2u);
        const float s0 = __low2float(s2), s1 = __high2float(s2);
        const uint32_t words[4] = {pv.x, pv.y, pv.z, pv.w};
        float wv[32];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            uint32_t h[4];
            e2m1x8_to_f16x2(words[t], h);
            const float sc = t < 2 ? s0 : s1;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const __half2 q = *reinterpret_cast<const __half2 *>(&h[i]);
                wv[8 * t + 2 * i] = __low2float(q) * sc;
                wv[8 * t + 2 * i + 1] = __high2float(q) * sc;
            }
        }
#pragma unroll
        for (int r = 0; r < kMaxRows; ++r) {
            if (r < rows) {
                const uint16_t *xr = x + (size_t)r * H + base;
                float a = acc[r];
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const uint4 xv = *reinterpret_cast<const uint4 *>(xr + 8 * v);
                    a = fmaf(bf16_lo(xv.x), wv[8 * v + 0], a);
                    a = fmaf(bf16_hi(xv.x), wv[8 * v + 1], a);
                    a = fmaf(bf16_lo(xv.y), wv[8 * v + 2], a);
                    a = fmaf(bf16_hi(xv.y), wv[8 * v + 3], a);
                    a = fmaf(bf16_lo(xv.z), wv[8 * v + 4], a);
                    a = fmaf(bf16_hi(xv.z), wv[8 * v + 5], a);
                    a = fmaf(bf16_lo(xv.w), wv[8 * v + 6], a);
                    a = fmaf(bf16_hi(xv.w), wv[8 * v + 7], a);
                }
                acc[r] = a;
            }
        }
    }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
// ---------------------------------------------------------------------------
// Route kernel
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(kRouteWarps * 32)
    moe_route_kernel(const RouteParams p) {
    __shared__ int32_t s_ids[kMaxIds];
    __shared__ float s_wts[kMaxIds];
    __shared__ int s_last;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * kRouteWarps + warp;   // router row of this warp
    const bool gate_row = p.has_shared && p.shared_gated;
    const int nrow = p.E + (gate_row ? 1 : 0);
    const int H = p.H;

    // Router weights are constant: start pulling this warp's row into L2
    // before waiting for the producer of x.
    if (row < nrow && lane == 0) {
        if (row == p.E) {
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.sh_vec),
                         "r"((uint32_t)(H * 2))
                         : "memory");
        } else if (p.router_fmt == MOE_ROUTER_BF16) {
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                             p.router_bf16 + (size_t)row * H),
                         "r"((uint32_t)(H * 2))
                         : "memory");
        } else {
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                             p.router_fp4.packed + (size_t)row * (H / 2)),
                         "r"((uint32_t)(H / 2))
                         : "memory");
        }
    }
    pdl_trigger();
    pdl_wait();

    if (row < nrow) {
        float acc[kMaxRows];
#pragma unroll
        for (int r = 0; r < kMaxRows; ++r) acc[r] = 0.f;
        if (row == p.E) {
            dot_bf16_row(p.sh_vec, p.x, H, p.rows, lane, acc);
        } else if (p.router_fmt == MOE_ROUTER_BF16) {
            dot_bf16_row(p.router_bf16 + (size_t)row * H, p.x, H, p.rows, lane, acc);
        } else {
            dot_nvfp4_row(p.router_fp4.packed + (size_t)row * (H / 2),
                          p.router_fp4.scales + (size_t)row * (H / 16), p.x, H, p.rows, lane,
                          acc);
        }
#pragma unroll
        for (int r = 0; r < kMaxRows; ++r) {
            if (r < p.rows) {
                float v = warp_sum(acc[r]);
                if (lane == 0) {
                    if (row == p.E) {
                        p.ws.gate_val[r] = 1.f / (1.f + expf(-v));
                    } else {
                        if (p.router_fmt == MOE_ROUTER_NVFP4) v *= p.router_fp4.scale2;
                        p.ws.logits[(size_t)r * p.E + row] = v;
                        if (p.logits_out) p.logits_out[(size_t)r * p.E + row] = v;
                    }
                }
            }
        }
    }

    // Last block to finish runs the top-k and the union.
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned t = atomicAdd(&p.ws.hdr->route_ticket, 1u);
        s_last = (t == gridDim.x - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    const int E = p.E, k = p.k;
    if (warp < p.rows) {
        const int r = warp;
        warp_topk_row(p.ws.logits + (size_t)r * E, p.bias, E, k, p.scoring, p.norm, p.rsf,
                      s_ids + r * k, s_wts + r * k, lane);
        __syncwarp();
        for (int j = lane; j < k; j += 32) {
            const int id = s_ids[r * k + j];
            const float w = s_wts[r * k + j];
            p.ws.ids[(p.row_base + r) * k + j] = id;
            p.ws.wts[(p.row_base + r) * k + j] = w;
            if (p.ids_out) p.ids_out[r * k + j] = id;
            if (p.wts_out) p.wts_out[r * k + j] = w;
        }
    }
    if (threadIdx.x < kMaxRows && !(p.has_shared && p.shared_gated))
        p.ws.gate_val[threadIdx.x] = p.has_shared ? 1.f : 0.f;
    if (threadIdx.x == 0) p.ws.hdr->route_ticket = 0u;
}

// ---------------------------------------------------------------------------
// Union kernel: up to kCallIds ids, one thread per position
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(kCallIds) moe_union_kernel(const UnionParams p) {
    __shared__ int32_t s_ids[kCallIds];
    __shared__ int s_uidx[kCallIds];              // union index of each first occurrence
    __shared__ int s_wfirst[kCallIds / 32];       // first occurrences per warp
    __shared__ uint32_t s_mask[kCallIds];         // row mask of each union entry
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int k = p.k, n = p.rows * k;
    pdl_wait();
    // unused positions get distinct negative ids, so they never match
    const int id = t < n ? p.ids[t] : -1 - t;
    s_ids[t] = id;
    s_mask[t] = 0u;
    __syncthreads();
    // Pairwise scan in blocks of 64: the earliest position holding this id
    // (earlier blocks first, then this position's own block); per-row mode
    // keeps every position.
    int fq = t;
    if (!p.per_row_mode && t < n) {
        const int blk0 = (t / kMaxIds) * kMaxIds;
        for (int q = 0; q < blk0 && fq == t; ++q)
            if (s_ids[q] == id) fq = q;
        for (int q = blk0; q < t && fq == t; ++q)
            if (s_ids[q] == id) fq = q;
    }
    const bool first = t < n && fq == t;
    const unsigned bal = __ballot_sync(0xffffffffu, first);
    if (lane == 0) s_wfirst[warp] = __popc(bal);
    __syncthreads();
    int base = 0, U = 0;
#pragma unroll
    for (int w = 0; w < kCallIds / 32; ++w) {
        base += w < warp ? s_wfirst[w] : 0;
        U += s_wfirst[w];
    }
    if (first) s_uidx[t] = base + __popc(bal & ((1u << lane) - 1u));
    moe_union_table *ut = p.ws.uni;
    uint4 *us = reinterpret_cast<uint4 *>(&ut->uslot[0][0]);
    for (int i = t; i < (int)(sizeof(ut->uslot) / 16); i += kCallIds)
        us[i] = make_uint4(~0u, ~0u, ~0u, ~0u);
    __syncthreads();
    if (t < n) {
        const int u = s_uidx[fq];
        ut->slot2u[t] = (uint8_t)u;
        ut->uslot[u][t / k] = (uint8_t)(t % k);
        atomicOr(&s_mask[u], 1u << (t / k));
    }
    __syncthreads();
    if (first) {
        const int u = s_uidx[t];
        ut->expert[u] = id;
        ut->rowmask[u] = s_mask[u];
        if (p.has_tables) {
            PtrEntry e;
            if (id < 0 || id >= p.E) {
                record_fault(p.ws.hdr, MOE_DEV_BAD_EXPERT_ID, (uint32_t)t);
                e = PtrEntry{};
                e.expert = -1;
            } else {
                const moe_expert_table tb[3] = {p.gate, p.up, p.down};
                load_ptr_entry(tb, id, e, p.has_scales != 0);
                bool ok = true;
#pragma unroll
                for (int m = 0; m < 3; ++m) ok = ok && aligned16(e.packed[m]) && aligned16(e.scales[m]);
                if (!ok) {
                    record_fault(p.ws.hdr, MOE_DEV_MISALIGNED_PTR, (uint32_t)id);
                    e.expert = -1;
                }
            }
            p.ws.ptrs[u] = e;
        } else if (id < 0 || id >= p.E) {
            record_fault(p.ws.hdr, MOE_DEV_BAD_EXPERT_ID, (uint32_t)t);
        }
    }
    if (t == 0) {
        ut->num_union = U;
        ut->rows = p.rows;
        ut->top_k = k;
        ut->per_row_mode = p.per_row_mode;
        if (p.has_tables && p.has_shared) {
            PtrEntry e;
            const moe_nvfp4 *sm3[3] = {&p.sh_gate, &p.sh_up, &p.sh_down};
#pragma unroll
            for (int m = 0; m < 3; ++m) {
                e.packed[m] = sm3[m]->packed;
                e.scales[m] = sm3[m]->scales;
                e.scale2[m] = sm3[m]->scale2;
            }
            e.expert = kSharedEntry;
            p.ws.ptrs[kCallIds] = e;
        }
    }
    if (p.out) {   // the caller's copy of the table
        __syncthreads();
        const uint32_t *s = reinterpret_cast<const uint32_t *>(ut);
        uint32_t *d = reinterpret_cast<uint32_t *>(p.out);
        for (int i = t; i < (int)(sizeof(moe_union_table) / 4); i += kCallIds) d[i] = s[i];
    }
}

// ---------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------

static cudaLaunchAttribute pdl_attr() {
    cudaLaunchAttribute a;
    a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    a.val.programmaticStreamSerializationAllowed = 1;
    return a;
}

cudaError_t launch_route(const RouteParams &p, cudaStream_t stream) {
    const int nrow = p.E + ((p.has_shared && p.shared_gated) ? 1 : 0);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((nrow + kRouteWarps - 1) / kRouteWarps);
    cfg.blockDim = dim3(kRouteWarps * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {pdl_attr()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, moe_route_kernel, p);
}

cudaError_t launch_union(const UnionParams &p, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(kCallIds);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {pdl_attr()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, moe_union_kernel, p);
}

}  // namespace moe
