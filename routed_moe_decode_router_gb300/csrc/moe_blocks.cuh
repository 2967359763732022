// moe_blocks.cuh -- device building blocks shared by the route kernel and the
// layer kernel: warp top-k, pairwise-scan union, pointer entries, the NVFP4
// x f16 MMA on one 128-input chunk, token-row fragments, the stage-ring wait
// and the grid barrier.
#pragma once

#include "moe_device.cuh"

namespace moe {

// ---------------------------------------------------------------------------
// Pointer entries
// ---------------------------------------------------------------------------

// Pointer entry (gate, up, down matrices) of expert x from the expert tables.
// (has_scales = 0: FP8 and BF16 experts, whose tables may hold no scale
// arrays; the entry's scale pointers are then NULL and never read.)
__device__ __forceinline__ void load_ptr_entry(const moe_expert_table *tabs, int x, PtrEntry &e,
                                               bool has_scales) {
#pragma unroll
    for (int m = 0; m < 3; ++m) {
        e.packed[m] = ld_cg(tabs[m].packed + x);
        e.scales[m] = has_scales ? ld_cg(tabs[m].scales + x) : nullptr;
        e.scale2[m] = ld_cg(tabs[m].scale2 + x);
    }
    e.expert = x;
}

__device__ __forceinline__ bool aligned16(const void *p) {
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

// ---------------------------------------------------------------------------
// Top-k of one token row (one warp)
// ---------------------------------------------------------------------------
//
// Selection key (forward_token_major.rs: moe_topk_softmax_batched /
// moe_topk_sigmoid_batched): the logit for softmax scoring (softmax is
// strictly increasing in it), sigmoid(logit) + correction bias for sigmoid
// scoring; largest key first, equal keys to the lower expert id, NaN keys
// rank lowest.  Weights: softmax -> exp(l_j - l_max) over the selected slots
// (norm_topk_prob) or over all experts; sigmoid -> sigmoid(l_j), normalised
// over the selected slots when norm_topk_prob, times routed_scaling_factor.
// All arithmetic is fp32 (expf, IEEE division); the sums are compensated.

// Error-free sum a + b = s + e (Knuth's TwoSum).
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e) {
    s = a + b;
    const float bb = s - a;
    e = (a - (s - bb)) + (b - bb);
}

// Compensated warp sum: every lane gets the same result, within about one
// rounding of the exact sum of the 32 lanes' (value, error) pairs.
__device__ __forceinline__ float warp_sum_compensated(float v, float c) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
        const float c2 = __shfl_xor_sync(0xffffffffu, c, o);
        float s, e;
        two_sum(v, v2, s, e);
        v = s;
        c = (c + c2) + e;
    }
    return v + c;
}

// Balanced trees over a register array (compile-time N): the largest value
// (fmaxf skips NaN, so the result does not depend on the order), the OR of
// bit masks, and the element at a run-time index (a select tree on its bits,
// so no local-memory indexing).
template <int N>
__device__ __forceinline__ float tree_fmax(const float (&a)[N]) {
    float t[N];
#pragma unroll
    for (int i = 0; i < N; ++i) t[i] = a[i];
#pragma unroll
    for (int w = N; w > 1; w = (w + 1) / 2) {
#pragma unroll
        for (int i = 0; i < w / 2; ++i) t[i] = fmaxf(t[2 * i], t[2 * i + 1]);
        if (w & 1) t[w / 2] = t[w - 1];
    }
    return t[0];
}

template <int N>
__device__ __forceinline__ uint32_t tree_or(const uint32_t (&a)[N]) {
    uint32_t t[N];
#pragma unroll
    for (int i = 0; i < N; ++i) t[i] = a[i];
#pragma unroll
    for (int w = N; w > 1; w = (w + 1) / 2) {
#pragma unroll
        for (int i = 0; i < w / 2; ++i) t[i] = t[2 * i] | t[2 * i + 1];
        if (w & 1) t[w / 2] = t[w - 1];
    }
    return t[0];
}

template <int N>
__device__ __forceinline__ float tree_pick(const float (&a)[N], int idx) {
    float t[N];
#pragma unroll
    for (int i = 0; i < N; ++i) t[i] = a[i];
#pragma unroll
    for (int w = N, bit = 0; w > 1; w = (w + 1) / 2, ++bit) {
        const bool hi = (idx >> bit) & 1;
#pragma unroll
        for (int i = 0; i < w / 2; ++i) t[i] = hi ? t[2 * i + 1] : t[2 * i];
        if (w & 1) t[w / 2] = t[w - 1];
    }
    return t[0];
}

// Each lane holds the keys of experts lane + 32 * i (i < NK * NL, so
// E <= 32 * NK * NL) in registers, loaded once.  A selection round takes
// every lane's best key with an fp32 max tree, the warp's best with one
// unsigned max reduction over an order-preserving form of the key, and the
// lowest expert id holding it with one unsigned min reduction; the lane
// holding that expert retires it (its key becomes NaN, which fmaxf skips).
// No sort and no predicate chains, so the rounds are short.
template <int NK, int NL>
__device__ __forceinline__ void warp_topk_row_nk(const float *lg, const float *bias, int E, int k,
                                                 int scoring, int norm, float rsf,
                                                 int32_t *ids_out, float *wts_out, int lane) {
    const unsigned FULL = 0xffffffffu;
    const bool sigm = scoring == MOE_SCORING_SIGMOID;
    constexpr int N = NK * NL;   // candidates per lane: experts lane + 32 * i
    float key[N], v[N];
    // every load first (clamped index, no branch between them), so one
    // memory latency covers them
#pragma unroll
    for (int i = 0; i < N; ++i) v[i] = ld_cg(lg + min(lane + 32 * i, E - 1));
    if (sigm) {
#pragma unroll
        for (int i = 0; i < N; ++i) key[i] = bias[min(lane + 32 * i, E - 1)];
    }
#pragma unroll
    for (int i = 0; i < N; ++i) {
        float kv;
        if (sigm) {
            v[i] = 1.f / (1.f + expf(-v[i]));
            kv = v[i] + key[i];
        } else {
            kv = v[i];
        }
        if (kv != kv) kv = -INFINITY;   // a NaN key ranks lowest
        kv += 0.f;                       // -0 ranks as +0
        // NaN marks an empty candidate: fmaxf ignores it and it equals nothing
        key[i] = lane + 32 * i < E ? kv : __int_as_float(0x7fffffff);
    }
    int my_id0 = 0, my_id1 = 0;     // expert of slots lane and lane + 32
    float my_v0 = 0.f, my_v1 = 0.f; // its logit (softmax) or sigmoid (sigmoid scoring)
    // With 16 or more candidates per lane the round's three linear chains
    // (max, lowest matching slot, the winner's value) are balanced trees;
    // with fewer they are short enough as they are.
    constexpr bool kTrees = N >= 16;
    for (int j = 0; j < k; ++j) {
        // this lane's best key (a max tree, no predicates)
        float m = key[0];
        if constexpr (kTrees) {
            m = tree_fmax<N>(key);
        } else {
#pragma unroll
            for (int i = 1; i < N; ++i) m = fmaxf(m, key[i]);
        }
        // order-preserving unsigned form; an all-empty lane (NaN) maps to 0
        uint32_t u = __float_as_uint(m);
        u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
        u = (m != m) ? 0u : u;
        const uint32_t mu = __reduce_max_sync(FULL, u);
        const float mk = __uint_as_float((mu & 0x80000000u) ? (mu & 0x7fffffffu) : ~mu);
        // the lowest expert id holding the best key (ties -> lower id): this
        // lane's lowest matching slot, then the warp's lowest id
        uint32_t cand = 0xffffffffu;
        if constexpr (kTrees) {
            uint32_t bits[N];
#pragma unroll
            for (int i = 0; i < N; ++i) bits[i] = key[i] == mk ? (1u << i) : 0u;
            const uint32_t hitmask = tree_or<N>(bits);
            cand = hitmask ? (uint32_t)(lane + 32 * (__ffs(hitmask) - 1)) : 0xffffffffu;
        } else {
#pragma unroll
            for (int i = N - 1; i >= 0; --i) cand = key[i] == mk ? (uint32_t)(lane + 32 * i) : cand;
        }
        const int bi = (int)__reduce_min_sync(FULL, cand);
        // its value, from the lane that holds it; that lane retires it
        float val = 0.f;
        if constexpr (kTrees) {
            val = tree_pick<N>(v, bi >> 5);
#pragma unroll
            for (int i = 0; i < N; ++i)
                key[i] = (lane + 32 * i == bi) ? __int_as_float(0x7fffffff) : key[i];
        } else {
#pragma unroll
            for (int i = 0; i < N; ++i) {
                const bool hit = lane + 32 * i == bi;
                val = hit ? v[i] : val;
                key[i] = hit ? __int_as_float(0x7fffffff) : key[i];
            }
        }
        const float bv = __shfl_sync(FULL, val, bi & 31);
        if (lane == (j & 31)) {
            if (j < 32) {
                my_id0 = bi;
                my_v0 = bv;
            } else {
                my_id1 = bi;
                my_v1 = bv;
            }
        }
    }
    // routing weights: lane j (and j + 32) owns slot j
    const float top = __shfl_sync(FULL, my_v0, 0);   // slot 0 holds the largest logit
    float w[2] = {0.f, 0.f};
#pragma unroll
    for (int h = 0; h < 2; ++h)
        if (lane + 32 * h < k) w[h] = sigm ? (h ? my_v1 : my_v0) : expf((h ? my_v1 : my_v0) - top);
    float denom = 1.f;
    if (norm) {
        float s, e;
        two_sum(w[0], w[1], s, e);
        denom = warp_sum_compensated(s, e);
    } else if (!sigm) {
        // softmax without renormalisation: the full denominator over all E
        float zsum = 0.f, zerr = 0.f;
        // the logits again (the values were kept in v), in expert order
#pragma unroll
        for (int i = 0; i < N; ++i) {
            float s, er;
            two_sum(zsum, lane + 32 * i < E ? expf(v[i] - top) : 0.f, s, er);
            zsum = s;
            zerr += er;
        }
        denom = warp_sum_compensated(zsum, zerr);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int j = lane + 32 * h;
        if (j < k) {
            ids_out[j] = h ? my_id1 : my_id0;
            float wj = w[h] / denom;
            if (sigm) wj *= rsf;
            wts_out[j] = wj;
        }
    }
}

// The same with the candidate count fixed at compile time (TK = the class of
// E: 0 for E <= 128, 1 for <= 256, 2 for <= 512, 3 for <= 1024).
template <int TK>
__device__ __forceinline__ void warp_topk_row_tk(const float *lg, const float *bias, int E, int k,
                                                 int scoring, int norm, float rsf,
                                                 int32_t *ids_out, float *wts_out, int lane) {
    if constexpr (TK == 0)
        warp_topk_row_nk<4, 1>(lg, bias, E, k, scoring, norm, rsf, ids_out, wts_out, lane);
    else if constexpr (TK == 1)
        warp_topk_row_nk<8, 1>(lg, bias, E, k, scoring, norm, rsf, ids_out, wts_out, lane);
    else if constexpr (TK == 2)
        warp_topk_row_nk<16, 1>(lg, bias, E, k, scoring, norm, rsf, ids_out, wts_out, lane);
    else
        warp_topk_row_nk<16, 2>(lg, bias, E, k, scoring, norm, rsf, ids_out, wts_out, lane);
}

__device__ __forceinline__ void warp_topk_row(const float *lg, const float *bias, int E, int k,
                                              int scoring, int norm, float rsf, int32_t *ids_out,
                                              float *wts_out, int lane) {
    if (E <= 128)
        warp_topk_row_nk<4, 1>(lg, bias, E, k, scoring, norm, rsf, ids_out, wts_out, lane);
    else if (E <= 256)
        warp_topk_row_nk<8, 1>(lg, bias, E, k, scoring, norm, rsf, ids_out, wts_out, lane);
    else if (E <= 512)
        warp_topk_row_nk<16, 1>(lg, bias, E, k, scoring, norm, rsf, ids_out, wts_out, lane);
    else
        warp_topk_row_nk<16, 2>(lg, bias, E, k, scoring, norm, rsf, ids_out, wts_out, lane);
}

// ---------------------------------------------------------------------------
// Union + pointer table (one warp)
// ---------------------------------------------------------------------------

struct UnionSrc {
    int E, k, rows, per_row_mode, has_tables, has_shared, has_scales;
    moe_expert_table gate, up, down;
    moe_nvfp4 sh_gate, sh_up, sh_down;
};

// Union of the rows * k <= 64 ids of one sub-chunk in s_ids (position p =
// row * k + slot) by pairwise scan (page "Function forward_moe", RETRACTED
// note): position p
// opens a union entry when no earlier position holds the same id; entries
// keep first-occurrence order; no sort.  Lane l holds positions l and l + 32;
// the comparisons against earlier positions run on registers (warp match
// within a half, shuffles across the halves).  Writes the table and, with
// has_tables, the pointer entry of every union expert plus the shared expert
// at kSharedEntry.  `ut` and `ptrs` may point to shared or global memory;
// s_mask is 64 words of scratch shared memory.  All 32 lanes of one warp
// call it.
__device__ inline void build_union(const UnionSrc &src, const int32_t *s_ids, uint32_t *s_mask,
                                   ChunkUnion *ut, PtrEntry *ptrs, WsHeader *hdr, int lane) {
    const unsigned FULL = 0xffffffffu;
    const int n = src.rows * src.k;
    const int p0 = lane, p1 = lane + 32;
    // unused positions get distinct negative ids, so they never match
    const int id0 = p0 < n ? s_ids[p0] : -1 - p0;
    const int id1 = p1 < n ? s_ids[p1] : -1 - p1;
    // the pointer entries of both positions' experts are loaded first (from
    // a clamped id), so their memory latency overlaps the scan below
    PtrEntry pe[2];
    if (src.has_tables) {
        const moe_expert_table tb[3] = {src.gate, src.up, src.down};
        load_ptr_entry(tb, min(max(id0, 0), src.E - 1), pe[0], src.has_scales);
        if (n > 32) load_ptr_entry(tb, min(max(id1, 0), src.E - 1), pe[1], src.has_scales);
    }
    const unsigned below = (1u << lane) - 1u;
    unsigned eq0, eq1, cross = 0;   // same-id lanes: half 0 for id0, half 1 for id1, half 0 for id1
    if (src.per_row_mode) {
        eq0 = 1u << lane;
        eq1 = 1u << lane;
    } else {
        eq0 = __match_any_sync(FULL, id0);
        eq1 = 1u << lane;   // positions >= n hold distinct negative ids
        if (n > 32) {       // warp-uniform
            eq1 = __match_any_sync(FULL, id1);
#pragma unroll
            for (int q = 0; q < 32; ++q) cross |= (__shfl_sync(FULL, id0, q) == id1 ? 1u : 0u) << q;
        }
    }
    const bool first0 = p0 < n && (eq0 & below) == 0;
    const bool first1 = p1 < n && cross == 0 && (eq1 & below) == 0;
    const unsigned f0 = __ballot_sync(FULL, first0);
    const unsigned f1 = __ballot_sync(FULL, first1);
    const int U = __popc(f0) + __popc(f1);
    const int uidx0 = __popc(f0 & below);
    const int uidx1 = __popc(f0) + __popc(f1 & below);
    // union index of every position: that of its first occurrence (every
    // lane runs every shuffle: a full-mask shuffle must not diverge)
    const int u0 = __shfl_sync(FULL, uidx0, __ffs(eq0) - 1);
    const int u1_cross = __shfl_sync(FULL, uidx0, cross ? __ffs(cross) - 1 : lane);
    const int u1_half = __shfl_sync(FULL, uidx1, __ffs(eq1) - 1);
    const int u1 = cross ? u1_cross : u1_half;
    s_mask[lane] = 0u;
    s_mask[lane + 32] = 0u;
    for (int i = lane; i < kMaxIds * kMaxRows; i += 32) (&ut->uslot[0][0])[i] = 0xFF;
    __syncwarp();
    const int k = src.k;
    if (p0 < n) {
        ut->slot2u[p0] = (uint8_t)u0;
        ut->uslot[u0][p0 / k] = (uint8_t)(p0 % k);
        atomicOr(&s_mask[u0], 1u << (p0 / k));
    }
    if (p1 < n) {
        ut->slot2u[p1] = (uint8_t)u1;
        ut->uslot[u1][p1 / k] = (uint8_t)(p1 % k);
        atomicOr(&s_mask[u1], 1u << (p1 / k));
    }
    __syncwarp();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const bool first = h ? first1 : first0;
        if (!first) continue;
        const int p = h ? p1 : p0;
        const int u = h ? uidx1 : uidx0;
        const int x = h ? id1 : id0;
        ut->expert[u] = x;
        ut->rowmask[u] = (uint8_t)s_mask[u];
        if (src.has_tables) {
            PtrEntry e;
            if (x < 0 || x >= src.E) {
                record_fault(hdr, MOE_DEV_BAD_EXPERT_ID, (uint32_t)p);
                e = PtrEntry{};
                e.expert = -1;
            } else {
                e = pe[h];
                bool ok = true;
#pragma unroll
                for (int m = 0; m < 3; ++m)
                    ok = ok && aligned16(e.packed[m]) && aligned16(e.scales[m]);
                if (!ok) {
                    record_fault(hdr, MOE_DEV_MISALIGNED_PTR, (uint32_t)x);
                    e.expert = -1;
                }
            }
            ptrs[u] = e;
        } else if (x < 0 || x >= src.E) {
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

// The union of ONE row (its k <= 64 distinct top-k ids): entry p is slot p,
// row mask 1; the same table and pointer entries build_union gives for one
// row, without the pairwise scan (the one-row layer form, whose code is
// kept small).  All 32 lanes of one warp call it.
__device__ inline void build_union_one_row(const UnionSrc &src, const int32_t *s_ids,
                                           ChunkUnion *ut, PtrEntry *ptrs, WsHeader *hdr,
                                           int lane) {
    const int n = src.k;
    const moe_expert_table tb[3] = {src.gate, src.up, src.down};
    for (int i = lane; i < kMaxIds * kMaxRows; i += 32) (&ut->uslot[0][0])[i] = 0xFF;
    __syncwarp();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int p = lane + 32 * h;
        if (p >= n) continue;
        const int x = s_ids[p];
        ut->expert[p] = x;
        ut->rowmask[p] = 1u;
        ut->slot2u[p] = (uint8_t)p;
        ut->uslot[p][0] = (uint8_t)p;
        PtrEntry e;
        if (x < 0 || x >= src.E) {
            record_fault(hdr, MOE_DEV_BAD_EXPERT_ID, (uint32_t)p);
            e = PtrEntry{};
            e.expert = -1;
        } else {
            load_ptr_entry(tb, x, e, src.has_scales);
            bool ok = true;
#pragma unroll
            for (int m = 0; m < 3; ++m) ok = ok && aligned16(e.packed[m]) && aligned16(e.scales[m]);
            if (!ok) {
                record_fault(hdr, MOE_DEV_MISALIGNED_PTR, (uint32_t)x);
                e.expert = -1;
            }
        }
        ptrs[p] = e;
    }
    if (lane == 0) {
        if (src.has_shared) {
            PtrEntry e;
            const moe_nvfp4 *sm3[3] = {&src.sh_gate, &src.sh_up, &src.sh_down};
#pragma unroll
            for (int m = 0; m < 3; ++m) {
                e.packed[m] = sm3[m]->packed;
                e.scales[m] = sm3[m]->scales;
                e.scale2[m] = sm3[m]->scale2;
            }
            e.expert = kSharedEntry;
            ptrs[kSharedEntry] = e;
        }
        ut->rows = 1;
        ut->top_k = src.k;
        ut->per_row_mode = src.per_row_mode;
        ut->num_union = n;
    }
}

// ---------------------------------------------------------------------------
// NVFP4 x f16 MMA on one 128-input chunk of a 16-row tile
// ---------------------------------------------------------------------------
//
// Lane (g = lane/4, q = lane%4) reads 16 bytes (32 inputs) of rows g and g+8
// at input offset q*32 inside the chunk, plus their two E4M3 scales; MMA
// step s (0..7) uses inputs 4s..4s+3 of that slice: logical k (2q, 2q+1) <-
// inputs (4s, 4s+1) and (2q+8, 2q+9) <- (4s+2, 4s+3).  The B fragments hold
// the token rows at the same inputs.  E2M1 x E4M3 is exact in f16.  Even
// steps accumulate into d0, odd steps into d1 (two independent MMA chains);
// the caller adds d0 + d1 in that order.
__device__ __forceinline__ void chunk_mma(const uint8_t *pk, const uint8_t *sc, int row_bytes,
                                          int sc_row_bytes, int c, int g, int q,
                                          const uint32_t (&b)[8][2], float (&d0)[4],
                                          float (&d1)[4]) {
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
        mma_f16_16816(d0, ha[0], hb[0], ha[1], hb[1], b[2 * t][0], b[2 * t][1]);
        mma_f16_16816(d1, ha[2], hb[2], ha[3], hb[3], b[2 * t + 1][0], b[2 * t + 1][1]);
    }
}

// chunk_mma for FP8 expert tiles (one E4M3 code per weight, row_bytes = K,
// no block scales): lane (g, q) reads the 32 codes of rows g and g+8 at
// input offset q*32 of the chunk (two 16-byte loads a row); inputs 8t .. 8t+7
// are bytes 8t .. 8t+7, converted pairwise (exact) into the same f16x2 order
// that e2m1x8_to_f16x2 gives, so the MMA steps and B fragments are those of
// chunk_mma.
__device__ __forceinline__ void chunk_mma_fp8(const uint8_t *pk, int row_bytes, int c, int g,
                                              int q, const uint32_t (&b)[8][2], float (&d0)[4],
                                              float (&d1)[4]) {
    const uint4 *ra = reinterpret_cast<const uint4 *>(pk + g * row_bytes + c * 128 + q * 32);
    const uint4 *rb = reinterpret_cast<const uint4 *>(pk + (g + 8) * row_bytes + c * 128 + q * 32);
    const uint4 a01[2] = {ra[0], ra[1]};
    const uint4 b01[2] = {rb[0], rb[1]};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const uint4 &ua = a01[t >> 1], &ub = b01[t >> 1];
        const uint32_t wa0 = (t & 1) ? ua.z : ua.x, wa1 = (t & 1) ? ua.w : ua.y;
        const uint32_t wb0 = (t & 1) ? ub.z : ub.x, wb1 = (t & 1) ? ub.w : ub.y;
        const uint32_t ha[4] = {e4m3x2_to_f16x2(wa0 & 0xFFFFu), e4m3x2_to_f16x2(wa0 >> 16),
                                e4m3x2_to_f16x2(wa1 & 0xFFFFu), e4m3x2_to_f16x2(wa1 >> 16)};
        const uint32_t hb[4] = {e4m3x2_to_f16x2(wb0 & 0xFFFFu), e4m3x2_to_f16x2(wb0 >> 16),
                                e4m3x2_to_f16x2(wb1 & 0xFFFFu), e4m3x2_to_f16x2(wb1 >> 16)};
        mma_f16_16816(d0, ha[0], hb[0], ha[1], hb[1], b[2 * t][0], b[2 * t][1]);
        mma_f16_16816(d1, ha[2], hb[2], ha[3], hb[3], b[2 * t + 1][0], b[2 * t + 1][1]);
    }
}

// chunk_mma for BF16 expert tiles (row_bytes = 2K): lane (g, q) reads the 32
// bf16 weights of rows g and g+8 at input offset q*32 (four 16-byte loads a
// row), which are already the A fragments of bf16 x bf16 MMAs; the B
// fragments hold the token rows as raw bf16 (load_b with RAW).
__device__ __forceinline__ void chunk_mma_bf16(const uint8_t *pk, int row_bytes, int c, int g,
                                               int q, const uint32_t (&b)[8][2], float (&d0)[4],
                                               float (&d1)[4]) {
    const uint4 *ra = reinterpret_cast<const uint4 *>(pk + g * row_bytes + c * 256 + q * 64);
    const uint4 *rb = reinterpret_cast<const uint4 *>(pk + (g + 8) * row_bytes + c * 256 + q * 64);
    uint4 wa[4], wb[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        wa[t] = ra[t];
        wb[t] = rb[t];
    }
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        mma_bf16_16816(d0, wa[t].x, wb[t].x, wa[t].y, wb[t].y, b[2 * t][0], b[2 * t][1]);
        mma_bf16_16816(d1, wa[t].z, wb[t].z, wa[t].w, wb[t].w, b[2 * t + 1][0], b[2 * t + 1][1]);
    }
}

// Expert formats: 0 NVFP4, 1 FP8 (E4M3 per weight), 2 BF16.  Bytes of one
// tile row of K inputs, and of its block scales.
template <int FMT>
__host__ __device__ constexpr uint32_t fmt_row_bytes(uint32_t K) {
    return FMT == 0 ? K / 2 : (FMT == 1 ? K : 2 * K);
}
template <int FMT>
__host__ __device__ constexpr uint32_t fmt_scale_row_bytes(uint32_t K) {
    return FMT == 0 ? K / 16 : 0;
}

// One 128-input chunk of a 16-row tile in the expert format FMT (the scale
// arguments are unused by FP8 and BF16).
template <int FMT>
__device__ __forceinline__ void chunk_mma_t(const uint8_t *pk, const uint8_t *sc, int row_bytes,
                                            int sc_row_bytes, int c, int g, int q,
                                            const uint32_t (&b)[8][2], float (&d0)[4],
                                            float (&d1)[4]) {
    if constexpr (FMT == 0)
        chunk_mma(pk, sc, row_bytes, sc_row_bytes, c, g, q, b, d0, d1);
    else if constexpr (FMT == 1)
        chunk_mma_fp8(pk, row_bytes, c, g, q, b, d0, d1);
    else
        chunk_mma_bf16(pk, row_bytes, c, g, q, b, d0, d1);
}

// The one-row CUDA-core variant of chunk_mma (one token row, column 0): the
// same lane data (rows g and g+8, inputs q*32..+31 of the chunk, their two
// block scales) and the same B fragments, whose every lane holds token row
// 0 (load_b with ROW0) scaled so that its largest magnitude lies in
// [2^8, 2^9).  Each 16-input block's eight f16x2 products are summed in f16
// (no partial can exceed 8 * 6 * 2^9 < 65504), the block sums are scaled in
// fp32, and the four lanes of a row are added by shuffles (q order fixed by
// the butterfly).  ra / rb receive the chunk's dot products of rows g and
// g+8 with the (scaled) token row.
__device__ __forceinline__ void chunk_gemv(const uint8_t *pk, const uint8_t *sc, int row_bytes,
                                           int sc_row_bytes, int c, int g, int q,
                                           const uint32_t (&b)[8][2], float &ra, float &rb) {
    const uint4 wa = *reinterpret_cast<const uint4 *>(pk + g * row_bytes + c * 64 + q * 16);
    const uint4 wb =
        *reinterpret_cast<const uint4 *>(pk + (g + 8) * row_bytes + c * 64 + q * 16);
    const uint32_t sa = *reinterpret_cast<const uint16_t *>(sc + g * sc_row_bytes + c * 8 + q * 2);
    const uint32_t sb =
        *reinterpret_cast<const uint16_t *>(sc + (g + 8) * sc_row_bytes + c * 8 + q * 2);
    const uint32_t wA[4] = {wa.x, wa.y, wa.z, wa.w};
    const uint32_t wB[4] = {wb.x, wb.y, wb.z, wb.w};
    __half2 acc[2][2];   // [row g / g+8][block 0 / 1]
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int k = 0; k < 2; ++k) acc[r][k] = __float2half2_rn(0.f);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        uint32_t ha[4], hb[4];
        e2m1x8_to_f16x2(wA[t], ha);
        e2m1x8_to_f16x2(wB[t], hb);
        const uint32_t xv[4] = {b[2 * t][0], b[2 * t][1], b[2 * t + 1][0], b[2 * t + 1][1]};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __half2 x2 = *reinterpret_cast<const __half2 *>(&xv[i]);
            acc[0][t >> 1] = __hfma2(*reinterpret_cast<const __half2 *>(&ha[i]), x2, acc[0][t >> 1]);
            acc[1][t >> 1] = __hfma2(*reinterpret_cast<const __half2 *>(&hb[i]), x2, acc[1][t >> 1]);
        }
    }
    const uint32_t fa = e4m3x2_to_f16x2(sa), fb = e4m3x2_to_f16x2(sb);
    const float2 sca = __half22float2(*reinterpret_cast<const __half2 *>(&fa));
    const float2 scb = __half22float2(*reinterpret_cast<const __half2 *>(&fb));
    const float2 a0 = __half22float2(acc[0][0]), a1 = __half22float2(acc[0][1]);
    const float2 b0 = __half22float2(acc[1][0]), b1 = __half22float2(acc[1][1]);
    float x = (a0.x + a0.y) * sca.x + (a1.x + a1.y) * sca.y;
    float y = (b0.x + b0.y) * scb.x + (b1.x + b1.y) * scb.y;
    x += __shfl_xor_sync(0xffffffffu, x, 1);
    y += __shfl_xor_sync(0xffffffffu, y, 1);
    x += __shfl_xor_sync(0xffffffffu, x, 2);
    y += __shfl_xor_sync(0xffffffffu, y, 2);
    ra = x;
    rb = y;
}

// B fragments of one token-row matrix (x or h) for this warp's chunks
// (chunk c = warp + nwarps*m): lane (n = lane/4, q = lane%4) takes row n's 32
// inputs at c*128 + q*32, in one pass of L2 loads; rows outside `mask` are
// zero.  The bf16 values are scaled by 2^e (e per row, from the largest
// magnitude over this warp's chunks) and converted to f16 in place.  inv0 /
// inv1 receive 2^-e of the D columns 2q and 2q+1.
//
// With ROW0 (the one-row CUDA-core variant) every lane takes token row 0, its
// largest magnitude goes to [2^8, 2^9) instead, and inv0 = inv1 = 2^-e.
// With RAW (BF16 expert tiles) the bf16 values stay as they are and
// inv0 = inv1 = 1.
template <int MAXC, bool ROW0 = false, bool RAW = false>
__device__ __forceinline__ void load_b(const uint16_t *rows_base, size_t row_stride,
                                       uint32_t mask, int nchunk, int warp, int nwarps,
                                       int lane, uint32_t (&b)[MAXC][8][2], float &inv0,
                                       float &inv1) {
    const int n = ROW0 ? 0 : lane >> 2, q = lane & 3;
    const bool on = (mask >> n) & 1u;
    // every load first, from a clamped address (row 0 when the row is off,
    // the last chunk when the chunk is past the end), then zero the unused
    const int nrow = on ? n : 0;
#pragma unroll
    for (int m = 0; m < MAXC; ++m) {
        const int c = min(warp + nwarps * m, nchunk - 1);
        const uint16_t *src = rows_base + (size_t)nrow * row_stride + c * kChunk + q * 32;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const uint4 xv = ld_cg_v4(src + 8 * v);
            b[m][2 * v][0] = xv.x;
            b[m][2 * v][1] = xv.y;
            b[m][2 * v + 1][0] = xv.z;
            b[m][2 * v + 1][1] = xv.w;
        }
    }
#pragma unroll
    for (int m = 0; m < MAXC; ++m) {
        const bool live = on && warp + nwarps * m < nchunk;
#pragma unroll
        for (int s2 = 0; s2 < 8; ++s2) {
            b[m][s2][0] = live ? b[m][s2][0] : 0u;
            b[m][s2][1] = live ? b[m][s2][1] : 0u;
        }
    }
    if constexpr (RAW) {
        inv0 = inv1 = 1.f;
        return;
    }
    float mx = 0.f;
#pragma unroll
    for (int m = 0; m < MAXC; ++m)
#pragma unroll
        for (int s = 0; s < 8; ++s)
#pragma unroll
            for (int h = 0; h < 2; ++h)
                mx = fmaxf(mx, fmaxf(fabsf(bf16_lo(b[m][s][h])), fabsf(bf16_hi(b[m][s][h]))));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const int e = ROW0 ? max(f16_block_exponent(mx) - 6, -126) : f16_block_exponent(mx);
    const float up = exp2i(e);
#pragma unroll
    for (int m = 0; m < MAXC; ++m)
#pragma unroll
        for (int s = 0; s < 8; ++s)
#pragma unroll
            for (int h = 0; h < 2; ++h)
                b[m][s][h] = pack_f16x2(bf16_lo(b[m][s][h]) * up, bf16_hi(b[m][s][h]) * up);
    const float inv = exp2i(-e);
    if (ROW0) {
        inv0 = inv1 = inv;
        return;
    }
    inv0 = __shfl_sync(0xffffffffu, inv, 8 * q);
    inv1 = __shfl_sync(0xffffffffu, inv, 8 * q + 4);
}

// D fragment (lane g, q: rows g / g+8, columns 2q / 2q+1) -> smem, column
// major [8 columns][16 rows], so that a column's 16 rows are contiguous.
// Index of (column col, row r) in a warp's 16-row x 8-column block of
// partial sums: column-major, rows XOR-swizzled in groups of four by the
// column pair, so the compute warps' scattered stores hit half as many banks
// twice and the epilogue's float4 reads (four rows of one column) stay
// contiguous and conflict-free.
__device__ __forceinline__ int partial_index(int col, int r) {
    return col * 16 + (r ^ (4 * ((col >> 1) & 3)));
}

// The MMA accumulator of one 16 x 8 tile (rows g and g + 8, columns 2q and
// 2q + 1) into a partial-sum block, undoing the column scales.
__device__ __forceinline__ void store_partial(float *dst, const float (&d)[4], int g, int q,
                                              float inv0, float inv1) {
    dst[partial_index(2 * q, g)] = d[0] * inv0;
    dst[partial_index(2 * q + 1, g)] = d[1] * inv1;
    dst[partial_index(2 * q, g + 8)] = d[2] * inv0;
    dst[partial_index(2 * q + 1, g + 8)] = d[3] * inv1;
}

// SiLU with the fast exponential and division (relative error about 1e-6,
// far below the bf16 rounding of the value it feeds).
__device__ __forceinline__ float silu(float x) { return __fdividef(x, 1.f + __expf(-x)); }

// ---------------------------------------------------------------------------
// Stage ring wait and grid barrier, both bounded
// ---------------------------------------------------------------------------

// Wait for the phase of `bar` with the given parity.  Gives up at once when
// the CTA's abort flag is set; after kWaitLimitCycles it records
// MOE_DEV_WAIT_TIMEOUT, sets the abort flag and gives up.
__device__ __forceinline__ bool ring_wait(uint64_t *bar, uint32_t parity, volatile int *abort,
                                          WsHeader *hdr, uint32_t info) {
    if (*abort) return false;
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort) return false;
        if (clock64() - t0 > kWaitLimitCycles) {
            *abort = 1;
            record_fault(hdr, MOE_DEV_WAIT_TIMEOUT, info);
            return false;
        }
        __nanosleep(64);   // leave issue slots to the warps that share the sub-partition
    }
    return true;
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// One arrival of this CTA at the grid barrier (called by one thread, after
// the CTA's own barrier, which orders the CTA's earlier writes before the
// release).  The counter only grows: arrival n belongs to episode n / G, and
// the episode ends when the counter reaches (episode + 1) * G, so there is
// no reset and no second atomic.  The spin is bounded: on timeout it records
// MOE_DEV_WAIT_TIMEOUT, sets the abort flag and returns false.  Requires
// every CTA of the grid to be resident at once (cooperative launch).
__device__ __forceinline__ bool grid_arrive_wait(unsigned long long *count, unsigned nblocks,
                                                 volatile int *abort, WsHeader *hdr,
                                                 uint32_t info) {
    unsigned long long old;
    asm volatile("atom.add.release.gpu.global.u64 %0, [%1], 1;"
                 : "=l"(old)
                 : "l"(count)
                 : "memory");
    const unsigned long long target = (old / nblocks + 1) * nblocks;
    if (ld_acquire_u64(count) >= target) return true;
    const long long t0 = clock64();
    while (ld_acquire_u64(count) < target) {
        if (*abort) return false;
        if (clock64() - t0 > kWaitLimitCycles) {
            *abort = 1;
            record_fault(hdr, MOE_DEV_WAIT_TIMEOUT, info);
            return false;
        }
        __nanosleep(20);
    }
    return true;
}

}  // namespace moe
