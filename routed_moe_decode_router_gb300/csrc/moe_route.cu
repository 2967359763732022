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
// on the logit, sigmoid scoring on sigmoid(logit) + correction bias.
//
// Union (page "Function forward_moe", RETRACTED and WIDENED notes): the
// rows * top_k <= 64 ids resolve in one warp by pairwise scan -- a position
// starts a union entry when no earlier position holds the same id -- with no
// sort and no copy to the host.  The same warp writes the device pointer
// table of the union experts (the forward_moe page's pointer-table upgrade
// path), which the expert kernels read.
#include <cuda_runtime.h>

#include "moe_device.cuh"

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
__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ---------------------------------------------------------------------------
// Union + pointer table (one warp)
// ---------------------------------------------------------------------------

struct UnionSrc {
    int E, k, rows, per_row_mode, has_tables, has_shared;
    moe_expert_table gate, up, down;
    moe_nvfp4 sh_gate, sh_up, sh_down;
};

__device__ __forceinline__ bool aligned16(const void *p) {
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

// s_ids: the rows * k ids in shared memory (position p = row * k + slot).
// Called by all 32 lanes of one warp.
__device__ void build_union(const UnionSrc &src, const int32_t *s_ids, uint8_t *s_uidx,
                            moe_union_table *ut, PtrEntry *ptrs, WsHeader *hdr, int lane) {
    const int n = src.rows * src.k;
    bool first[2];
    int id[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int p = lane + 32 * h;
        id[h] = p < n ? s_ids[p] : -1;
        bool f = p < n;
        if (f && !src.per_row_mode) {
            for (int q = 0; q < p; ++q) {
                if (s_ids[q] == id[h]) {
                    f = false;
                    break;
                }
            }
        }
        first[h] = f;
    }
    const unsigned lo = __ballot_sync(0xffffffffu, first[0]);
    const unsigned hi = __ballot_sync(0xffffffffu, first[1]);
    const unsigned below = (1u << lane) - 1u;
    const int U = __popc(lo) + __popc(hi);
    int uidx[2];
    uidx[0] = __popc(lo & below);
    uidx[1] = __popc(lo) + __popc(hi & below);
#pragma unroll
    for (int h = 0; h < 2; ++h)
        if (first[h]) s_uidx[lane + 32 * h] = (uint8_t)uidx[h];
    // clear the per-row slot table of every union entry
    for (int i = lane; i < kMaxIds * kMaxRows; i += 32) (&ut->uslot[0][0])[i] = 0xFF;
    __syncwarp();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int p = lane + 32 * h;
        if (p >= n) continue;
        int u;
        if (first[h]) {
            u = uidx[h];
        } else {
            int q = 0;
            while (s_ids[q] != id[h]) ++q;   // the first occurrence exists
            u = s_uidx[q];
        }
        ut->slot2u[p] = (uint8_t)u;
        ut->uslot[u][p / src.k] = (uint8_t)(p % src.k);
        if (!first[h]) continue;
        uint32_t mask = 0;
        if (src.per_row_mode) {
            mask = 1u << (p / src.k);
        } else {
            for (int q = 0; q < n; ++q)
                if (s_ids[q] == id[h]) mask |= 1u << (q / src.k);
        }
        ut->expert[u] = id[h];
        ut->rowmask[u] = (uint8_t)mask;
        if (src.has_tables) {
            PtrEntry e;
            const int x = id[h];
            if (x < 0 || x >= src.E) {
                record_fault(hdr, MOE_DEV_BAD_EXPERT_ID, (uint32_t)p);
                e = PtrEntry{};
                e.expert = -1;
            } else {
                const moe_expert_table *tb[3] = {&src.gate, &src.up, &src.down};
                bool ok = true;
#pragma unroll
                for (int m = 0; m < 3; ++m) {
                    e.packed[m] = tb[m]->packed[x];
                    e.scales[m] = tb[m]->scales[x];
                    e.scale2[m] = tb[m]->scale2[x];
                    ok = ok && aligned16(e.packed[m]) && aligned16(e.scales[m]);
                }
                e.expert = x;
                if (!ok) {
                    record_fault(hdr, MOE_DEV_MISALIGNED_PTR, (uint32_t)x);
                    e.expert = -1;
                }
            }
            ptrs[u] = e;
        } else if (id[h] < 0 || id[h] >= src.E) {
            record_fault(hdr, MOE_DEV_BAD_EXPERT_ID, (uint32_t)p);
        }
    }
    if (lane == 0) {
        if (src.has_tables && src.has_shared) {
            PtrEntry e;
            const moe_nvfp4 *sm[3] = {&src.sh_gate, &src.sh_up, &src.sh_down};
#pragma unroll
            for (int m = 0; m < 3; ++m) {
                e.packed[m] = sm[m]->packed;
                e.scales[m] = sm[m]->scales;
                e.scale2[m] = sm[m]->scale2;
            }
            e.expert = kSharedEntry;
            ptrs[kSharedEntry] = e;
        }
        ut->rows = src.rows;
        ut->top_k = src.k;
        ut->per_row_mode = src.per_row_mode;
        ut->num_union = U;
    }
}

// ---------------------------------------------------------------------------
// Route kernel
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(kRouteWarps * 32)
    moe_route_kernel(const RouteParams p) {
    __shared__ int32_t s_ids[kMaxIds];
    __shared__ uint8_t s_uidx[kMaxIds];
    __shared__ uint32_t s_taken[kMaxRows][MOE_MAX_EXPERTS / 32];
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
        const float *lg = p.ws.logits + (size_t)r * E;
        uint32_t *taken = s_taken[r];
        for (int i = lane; i < MOE_MAX_EXPERTS / 32; i += 32) taken[i] = 0u;
        __syncwarp();
        for (int j = 0; j < k; ++j) {
            float bk = -INFINITY;
            int bi = 0x7fffffff;
            for (int e = lane; e < E; e += 32) {
                if ((taken[e >> 5] >> (e & 31)) & 1u) continue;
                const float l = ld_cg(lg + e);
                float key = l;
                if (p.scoring == MOE_SCORING_SIGMOID) key = 1.f / (1.f + expf(-l)) + p.bias[e];
                if (key != key) key = -INFINITY;   // NaN ranks lowest
                if (key > bk || (key == bk && e < bi)) {
                    bk = key;
                    bi = e;
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ok = __shfl_xor_sync(0xffffffffu, bk, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                if (ok > bk || (ok == bk && oi < bi)) {
                    bk = ok;
                    bi = oi;
                }
            }
            if (lane == 0) {
                taken[bi >> 5] |= 1u << (bi & 31);
                s_ids[r * k + j] = bi;
            }
            __syncwarp();
        }
        // routing weights of the k selected experts
        const float top = ld_cg(lg + s_ids[r * k]);
        float val[2] = {0.f, 0.f};
        double part = 0.0;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int j = lane + 32 * h;
            if (j < k) {
                const float l = ld_cg(lg + s_ids[r * k + j]);
                val[h] = (p.scoring == MOE_SCORING_SOFTMAX) ? expf(l - top)
                                                            : 1.f / (1.f + expf(-l));
                part += (double)val[h];
            }
        }
        double denom = 1.0;
        if (p.norm) {
            denom = warp_sum_d(part);
        } else if (p.scoring == MOE_SCORING_SOFTMAX) {
            double z = 0.0;
            for (int e = lane; e < E; e += 32) z += (double)expf(ld_cg(lg + e) - top);
            denom = warp_sum_d(z);
        }
        const double scale = (p.scoring == MOE_SCORING_SIGMOID) ? (double)p.rsf : 1.0;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int j = lane + 32 * h;
            if (j < k) {
                const float w = (float)((double)val[h] / denom * scale);
                const int id = s_ids[r * k + j];
                p.ws.ids[r * k + j] = id;
                p.ws.wts[r * k + j] = w;
                if (p.ids_out) p.ids_out[r * k + j] = id;
                if (p.wts_out) p.wts_out[r * k + j] = w;
            }
        }
    }
    if (threadIdx.x < kMaxRows && !(p.has_shared && p.shared_gated))
        p.ws.gate_val[threadIdx.x] = p.has_shared ? 1.f : 0.f;
    __syncthreads();
    if (p.do_union && warp == 0) {
        UnionSrc src{E,      k,      p.rows, p.per_row_mode, 1,        p.has_shared,
                     p.gate, p.up,   p.down, p.sh_gate,      p.sh_up, p.sh_down};
        build_union(src, s_ids, s_uidx, p.ws.uni, p.ws.ptrs, p.ws.hdr, lane);
    }
    if (threadIdx.x == 0) p.ws.hdr->route_ticket = 0u;
}

// ---------------------------------------------------------------------------
// Union-only kernel (one warp)
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(32) moe_union_kernel(const UnionParams p) {
    __shared__ int32_t s_ids[kMaxIds];
    __shared__ uint8_t s_uidx[kMaxIds];
    const int lane = threadIdx.x;
    pdl_wait();
    const int n = p.rows * p.k;
    for (int i = lane; i < kMaxIds; i += 32) s_ids[i] = i < n ? p.ids[i] : -1;
    __syncwarp();
    UnionSrc src{p.E,    p.k,    p.rows, p.per_row_mode, p.has_tables, p.has_shared,
                 p.gate, p.up,   p.down, p.sh_gate,      p.sh_up,      p.sh_down};
    build_union(src, s_ids, s_uidx, p.ws.uni, p.ws.ptrs, p.ws.hdr, lane);
    __syncwarp();
    if (p.out) {
        const uint32_t *s = reinterpret_cast<const uint32_t *>(p.ws.uni);
        uint32_t *d = reinterpret_cast<uint32_t *>(p.out);
        __threadfence_block();
        for (int i = lane; i < (int)(sizeof(moe_union_table) / 4); i += 32) d[i] = s[i];
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
    cfg.blockDim = dim3(32);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {pdl_attr()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, moe_union_kernel, p);
}

}  // namespace moe
