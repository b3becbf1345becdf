// Batched lossless draft verification on GB300 (sm_103a).
//
// Method (restated from the pages):
//   * p = softmax(z_target / T), q = softmax(z_draft / T) over the full
//     vocabulary for every tested draft position ("UraionSpec", §2.1, eq.
//     (acceptance)).
//   * Draft token x_j is accepted when u_j * q(x_j) < p(x_j), i.e. with
//     probability min(1, p/q); the first rejection n ends the prefix.
//   * At a rejection the emitted token is drawn from the normalised residual
//     max(p_n - q_n, 0); if every tested draft was accepted, a bonus token is
//     drawn from p of target row ell ("breaking down dspark and its lineage",
//     section "Preserving the target distribution during verification";
//     "AngelSpec" §1).
//   * T == 0 is greedy: accept while x_j is the target argmax.
//
// Kernel chain on the caller's stream (no host synchronisation; both kernels
// are programmatic dependent launches of the kernel before them, placed while
// it drains and waiting in griddepcontrol.wait before touching its results):
//   k_row_stats  persistent, one CTA per SM: the HBM pass.  Each CTA first
//                derives the needed rows from verify_len (target 0..ell, draft
//                0..ell-1).  Each warp then streams 4 KiB row chunks through its
//                own ring of shared-memory stages filled by 1-D bulk copies
//                (cp.async.bulk + mbarrier) and writes one partial per chunk:
//                (integer scale, sum of 2^(z*c - scale)) or (max, argmax).
//   k_finish     one thread-block cluster per request: validates the request,
//                merges chunk partials per row (exact power-of-two rescaling,
//                two-float sums), runs the accept tests with one warp ballot,
//                writes the accepted prefix; at T > 0 sums the draw weights of
//                the 1-2 draw rows per chunk across the cluster and draws the
//                token by inverse CDF over two-float prefixes (chunk totals,
//                then the chosen chunk's segments and elements).
#include <math.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include <cooperative_groups.h>

#include "specv_rowstats.cuh"
#include "specv_trace.h"

namespace cg = cooperative_groups;

namespace specv {

__device__ __forceinline__ bool in01(float u) { return u >= 0.0f && u < 1.0f; }

// =================================================================== accept

// Merge the chunk partials of one row.  T > 0: M = max of the chunks'
// integer scales, S = sum_c S_c * 2^(M_c - M) with exact power-of-two rescaling
// and a two-float accumulator.  T == 0: (max, lowest argmax).  Returns false
// for an invalid row.
template <bool GREEDY>
__device__ __forceinline__ bool merge_row(const float2* part, int nch, int lane, float& M, DF& S, int& arg) {
    // the first 4 * 32 partials are loaded at once (constant register slots);
    // longer rows continue in a loop
    constexpr int K = 4;
    float2 keep[K];
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int c = lane + 32 * k;
        keep[k] = c < nch ? part[c] : make_float2(-INFINITY, GREEDY ? __int_as_float(0x7fffffff) : 0.f);
    }
    if (GREEDY) {
        float best = -INFINITY;
        int ix = 0x7fffffff;
        bool bad = false;
        auto take = [&](float2 p) {
            const int i = __float_as_int(p.y);
            if (p.x != p.x) bad = true;
            else if (p.x > best || (p.x == best && i < ix)) { best = p.x; ix = i; }
        };
#pragma unroll
        for (int k = 0; k < K; ++k) take(keep[k]);
        for (int c = lane + 32 * K; c < nch; c += 32) take(part[c]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ob = __shfl_xor_sync(0xffffffffu, best, o);
            const int oi = __shfl_xor_sync(0xffffffffu, ix, o);
            if (ob > best || (ob == best && oi < ix)) { best = ob; ix = oi; }
        }
        bad = __any_sync(0xffffffffu, bad);
        M = best;
        arg = ix;
        S.hi = 1.f;
        S.lo = 0.f;
        return !bad && fabsf(best) <= 3.402823466e38f;
    }
    float m = -INFINITY;
#pragma unroll
    for (int k = 0; k < K; ++k) m = fmax_nan(m, keep[k].x);
    for (int c = lane + 32 * K; c < nch; c += 32) m = fmax_nan(m, part[c].x);
    m = warp_max_nan(m);
    M = m;
    arg = 0;
    if (m != m || m == -INFINITY) return false;
    DF acc = {0.f, 0.f};
    auto add = [&](float2 p) {
        if (p.x != -INFINITY) {
            // both scales are integer-valued: the rescale is an exact power of two
            const float d = p.x - m;
            const float v = p.y * pow2_f(d < -1000.f ? -1000 : (int)d);
            acc = df_add(acc, DF{v, 0.f});
        }
    };
#pragma unroll
    for (int k = 0; k < K; ++k) add(keep[k]);
    for (int c = lane + 32 * K; c < nch; c += 32) add(part[c]);
    S = warp_sum_df(acc);
    return S.hi > 0.f && S.hi <= 3.0e38f;
}

// p = e / (S.hi + S.lo) in fp32
__device__ __forceinline__ float div_df(float e, DF S) {
    const float q = e / S.hi;
    return fmaf(-q, S.lo / S.hi, q);
}

// ===================================================================== draw

// Weight of one element of the draw: the residual max(e_t - rho * e_d, 0)
// (both relative to their rows' scales, rho = S_t / S_d as a float pair) or
// the target weight e_t.  p_v - q_v = (e_t - rho * e_d) / S_t.
__device__ __forceinline__ float draw_weight(const ReqState& rs, float zt, float zd, float c_hi,
                                             float c_lo) {
    const float et = scaled_exp(zt, c_hi, c_lo, rs.M_t);
    if (rs.mode != 1) return et;
    const float ed = scaled_exp(zd, c_hi, c_lo, rs.M_d);
    return fmaxf(fmaf(-rs.rho_lo, ed, fmaf(-rs.rho_hi, ed, et)), 0.f);
}

template <int ES>
__device__ __forceinline__ float draw_weight_at(const ReqState& rs, const char* rt, const char* rd, int i,
                                                float c_hi, float c_lo) {
    return draw_weight(rs, load_logit<ES>(rt, i), rs.mode == 1 ? load_logit<ES>(rd, i) : 0.f, c_hi, c_lo);
}

// Sum of the weights of one 16-byte vector pair in element order.
template <int ES>
__device__ __forceinline__ float vec_weight_sum_ordered(const ReqState& rs, const uint4& t, const uint4& d,
                                                        float c_hi, float c_lo) {
    const uint32_t tw[4] = {t.x, t.y, t.z, t.w}, dw[4] = {d.x, d.y, d.z, d.w};
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        if (ES == 2) {
            s += draw_weight(rs, bf16_lo(tw[k]), bf16_lo(dw[k]), c_hi, c_lo);
            s += draw_weight(rs, bf16_hi(tw[k]), bf16_hi(dw[k]), c_hi, c_lo);
        } else {
            s += draw_weight(rs, __uint_as_float(tw[k]), __uint_as_float(dw[k]), c_hi, c_lo);
        }
    }
    return s;
}


// Lane segments of a chunk [e0, e1): lane l owns a contiguous run of
// elements.  A full, 16-byte-aligned chunk gives every lane kVecPerLane
// vectors (64 bf16 / 32 fp32 elements); any other chunk is split evenly.
template <int ES>
__device__ __forceinline__ bool chunk_full(const ReqState& rs, const char* rt, const char* rd, int e0, int e1) {
    return (e1 - e0) * ES == kChunkBytes && ((((uintptr_t)(rt + (size_t)e0 * ES)) & 15) == 0) &&
           (rs.mode != 1 || ((((uintptr_t)(rd + (size_t)e0 * ES)) & 15) == 0));
}

// The chunk can be read as whole 16-byte vectors in both rows (always true
// when the rows are 16-byte aligned and V * element size is a multiple of 16).
template <int ES>
__device__ __forceinline__ bool chunk_vec(const ReqState& rs, const char* rt, const char* rd, int e0, int e1) {
    return ((e1 - e0) * ES) % 16 == 0 && ((((uintptr_t)(rt + (size_t)e0 * ES)) & 15) == 0) &&
           (rs.mode != 1 || ((((uintptr_t)(rd + (size_t)e0 * ES)) & 15) == 0));
}

template <int ES>
__device__ __forceinline__ void seg_bounds(int e0, int e1, int lane, bool full, int& s0, int& s1) {
    const int seg = full ? kVecPerLane * (16 / ES) : (e1 - e0 + 31) / 32;
    s0 = min(e1, e0 + lane * seg);
    s1 = min(e1, s0 + seg);
}

// fp32 sum (in element order) of the draw weights over this lane's segment,
// and the last element with positive weight (-1 if none).
template <int ES>
__device__ __forceinline__ float seg_weight_sum(const ReqState& rs, const char* rt, const char* rd, int e0, int e1,
                                                bool full, int lane, float c_hi, float c_lo, int& lpos) {
    constexpr int EPV = 16 / ES;
    constexpr int HALF = kVecPerLane / 2;
    int s0, s1;
    seg_bounds<ES>(e0, e1, lane, full, s0, s1);
    float lsum = 0.f;
    lpos = -1;
    if (full) {
        const uint4* vt = (const uint4*)(rt + (size_t)s0 * ES);
        const uint4* vd = (const uint4*)(rd + (size_t)s0 * ES);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint4 tv[HALF], dv[HALF];
#pragma unroll
            for (int k = 0; k < HALF; ++k) {
                tv[k] = __ldg(vt + h * HALF + k);
                dv[k] = rs.mode == 1 ? __ldg(vd + h * HALF + k) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int k = 0; k < HALF; ++k) {
                const int base = s0 + (h * HALF + k) * EPV;
                const uint32_t tw[4] = {tv[k].x, tv[k].y, tv[k].z, tv[k].w};
                const uint32_t dw[4] = {dv[k].x, dv[k].y, dv[k].z, dv[k].w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if (ES == 2) {
                        const float w0 = draw_weight(rs, bf16_lo(tw[q]), bf16_lo(dw[q]), c_hi, c_lo);
                        const float w1 = draw_weight(rs, bf16_hi(tw[q]), bf16_hi(dw[q]), c_hi, c_lo);
                        lsum += w0;
                        if (w0 > 0.f) lpos = base + 2 * q;
                        lsum += w1;
                        if (w1 > 0.f) lpos = base + 2 * q + 1;
                    } else {
                        const float w0 =
                            draw_weight(rs, __uint_as_float(tw[q]), __uint_as_float(dw[q]), c_hi, c_lo);
                        lsum += w0;
                        if (w0 > 0.f) lpos = base + q;
                    }
                }
            }
        }
    } else {
        for (int i = s0; i < s1; ++i) {
            const float w = draw_weight_at<ES>(rs, rt, rd, i, c_hi, c_lo);
            lsum += w;
            if (w > 0.f) lpos = i;
        }
    }
    return lsum;
}

// The draw inside segment [seg0, seg1) (at most 64 elements) given the
// remainder rr: its elements spread over the warp (one or two per lane), an
// fp32 scan, the first element whose running weight exceeds rr; if rounding
// leaves none, the segment's last element with positive weight.
template <int ES>
__device__ __forceinline__ int seg_pick(const ReqState& rs, const char* rt, const char* rd, int seg0, int seg1,
                                        float rr, int lane, float c_hi, float c_lo) {
    const int epl = (seg1 - seg0 + 31) / 32;
    const int i0 = seg0 + lane * epl;
    const float w0 = i0 < seg1 ? draw_weight_at<ES>(rs, rt, rd, i0, c_hi, c_lo) : 0.f;
    const float w1 = (epl > 1 && i0 + 1 < seg1) ? draw_weight_at<ES>(rs, rt, rd, i0 + 1, c_hi, c_lo) : 0.f;
    const float part = w0 + w1;
    float incl = part;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, incl > rr);
    if (hit) {
        const int i = __ffs(hit) - 1;
        const int v = ((incl - part) + w0 > rr || epl == 1) ? i0 : i0 + 1;
        return __shfl_sync(0xffffffffu, v, i);
    }
    int lp = w1 > 0.f ? i0 + 1 : (w0 > 0.f ? i0 : -1);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lp = max(lp, __shfl_xor_sync(0xffffffffu, lp, o));
    return lp >= 0 ? lp : seg1 - 1;
}

// A full, aligned chunk is 8 "rounds" of 32 consecutive 16-byte vectors; in
// round k lane l holds vector 32k + l, so the rounds are contiguous runs of
// elements and every load is coalesced.  Per-round weight sums over the warp:
// lane l of the result holds the total of round l >> 2 (a transposing
// butterfly: 9 shuffles for 8 sums).
__device__ __forceinline__ float rounds_reduce(float (&v)[8], int lane) {
    // step xor 16: lanes < 16 keep rounds 0-3, others 4-7
    float a4[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float send = (lane & 16) ? v[k] : v[k + 4];
        const float got = __shfl_xor_sync(0xffffffffu, send, 16);
        a4[k] = ((lane & 16) ? v[k + 4] : v[k]) + got;
    }
    float a2[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const float send = (lane & 8) ? a4[k] : a4[k + 2];
        const float got = __shfl_xor_sync(0xffffffffu, send, 8);
        a2[k] = ((lane & 8) ? a4[k + 2] : a4[k]) + got;
    }
    const float send = (lane & 4) ? a2[0] : a2[1];
    float a1 = ((lane & 4) ? a2[1] : a2[0]) + __shfl_xor_sync(0xffffffffu, send, 4);
    a1 += __shfl_xor_sync(0xffffffffu, a1, 2);
    a1 += __shfl_xor_sync(0xffffffffu, a1, 1);
    return a1;
}

// Draw weights of a full chunk summed per round (fp32, element order inside a
// lane's vector); returns this lane's share of the round totals (see above).
// nvec: 16-byte vectors in the chunk (at most 256); vectors past it weigh 0.
template <int ES>
__device__ __forceinline__ float chunk_round_sums(const ReqState& rs, const char* rt, const char* rd, int e0,
                                                  int nvec, int lane, float c_hi, float c_lo) {
    constexpr int HALF = kVecPerLane / 2;
    const uint4* vt = (const uint4*)(rt + (size_t)e0 * ES);
    const uint4* vd = (const uint4*)(rd + (size_t)e0 * ES);
    // the second half's vectors are fetched while the first half is reduced
#pragma unroll
    for (int k = HALF; k < 2 * HALF; ++k) {
        const int i = 32 * k + lane;
        if (i < nvec) {
            asm volatile("prefetch.global.L1 [%0];" ::"l"(vt + i));
            if (rs.mode == 1) asm volatile("prefetch.global.L1 [%0];" ::"l"(vd + i));
        }
    }
    float r[8];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint4 tv[HALF], dv[HALF];
#pragma unroll
        for (int k = 0; k < HALF; ++k) {
            const int i = 32 * (h * HALF + k) + lane;
            tv[k] = make_uint4(0, 0, 0, 0);
            dv[k] = make_uint4(0, 0, 0, 0);
            if (i < nvec) {
                tv[k] = __ldg(vt + i);
                if (rs.mode == 1) dv[k] = __ldg(vd + i);
            }
        }
#pragma unroll
        for (int k = 0; k < HALF; ++k)
            r[h * HALF + k] = 32 * (h * HALF + k) + lane < nvec
                                  ? vec_weight_sum_ordered<ES>(rs, tv[k], dv[k], c_hi, c_lo) : 0.f;
    }
    return rounds_reduce(r, lane);
}

// The draw inside round k of a full chunk given the remainder rr: each lane
// takes its vector (8 bf16 / 4 fp32 elements), fp32 lane sums, a warp scan,
// then the crossing lane walks its elements; if rounding leaves no element,
// the round's last element with positive weight.
template <int ES>
__device__ __forceinline__ int round_pick(const ReqState& rs, const char* rt, const char* rd, int e0, int nvec,
                                          int k, float rr, int lane, float c_hi, float c_lo) {
    constexpr int EPV = 16 / ES;
    const bool in = 32 * k + lane < nvec;
    const uint4 t = in ? __ldcg((const uint4*)(rt + (size_t)e0 * ES) + 32 * k + lane) : make_uint4(0, 0, 0, 0);
    const uint4 d = (in && rs.mode == 1) ? __ldcg((const uint4*)(rd + (size_t)e0 * ES) + 32 * k + lane)
                                         : make_uint4(0, 0, 0, 0);
    const uint32_t tw[4] = {t.x, t.y, t.z, t.w}, dw[4] = {d.x, d.y, d.z, d.w};
    float w[EPV];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        if (ES == 2) {
            w[2 * q] = draw_weight(rs, bf16_lo(tw[q]), bf16_lo(dw[q]), c_hi, c_lo);
            w[2 * q + 1] = draw_weight(rs, bf16_hi(tw[q]), bf16_hi(dw[q]), c_hi, c_lo);
        } else {
            w[q] = draw_weight(rs, __uint_as_float(tw[q]), __uint_as_float(dw[q]), c_hi, c_lo);
        }
    }
    if (!in) {
#pragma unroll
        for (int e = 0; e < EPV; ++e) w[e] = 0.f;
    }
    float ls = 0.f;
    int lp = -1;
    const int base = e0 + (32 * k + lane) * EPV;
#pragma unroll
    for (int e = 0; e < EPV; ++e) {
        ls += w[e];
        if (w[e] > 0.f) lp = base + e;
    }
    float incl = ls;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, incl > rr);
    if (hit) {
        const int l = __ffs(hit) - 1;
        int v = -1;
        float cum = incl - ls;
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
            cum += w[e];
            if (v < 0 && cum > rr) v = base + e;
        }
        if (v < 0) v = lp >= 0 ? lp : base + EPV - 1;
        return __shfl_sync(0xffffffffu, v, l);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lp = max(lp, __shfl_xor_sync(0xffffffffu, lp, o));
    return lp >= 0 ? lp : e0 + min(nvec, 32 * k + 32) * EPV - 1;
}

// First lane (or element) where an inclusive two-float scan of nonnegative
// values exceeds the target; the exclusive prefix there.  Returns -1 if none.
__device__ __forceinline__ int scan_find(DF v, DF target, int lane, DF& excl) {
    const DF incl = warp_scan_df(v, lane);
    const bool over = incl.hi > target.hi || (incl.hi == target.hi && incl.lo > target.lo);
    const unsigned hit = __ballot_sync(0xffffffffu, over);
    if (!hit) return -1;
    const int l = __ffs(hit) - 1;
    DF e = df_add(incl, DF{-v.hi, -v.lo});
    excl.hi = __shfl_sync(0xffffffffu, e.hi, l);
    excl.lo = __shfl_sync(0xffffffffu, e.lo, l);
    return l;
}

// Inverse-CDF draw inside one chunk by a scan of its lane segments (one warp):
// the smallest element index whose running weight (from 0 at the chunk start)
// exceeds r; if none, the last element with positive weight.
template <int ES>
__device__ int chunk_pick(const ReqState& rs, const char* rt, const char* rd, int e0, int e1, DF r, int lane,
                          float c_hi, float c_lo) {
    const bool full = chunk_full<ES>(rs, rt, rd, e0, e1);
    int lpos;
    const float lsum = seg_weight_sum<ES>(rs, rt, rd, e0, e1, full, lane, c_hi, c_lo, lpos);
    DF excl;
    const int l = scan_find(DF{lsum, 0.f}, r, lane, excl);
    if (l < 0) {
        int lp = lpos;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lp = max(lp, __shfl_xor_sync(0xffffffffu, lp, o));
        return lp >= 0 ? lp : e1 - 1;
    }
    int s0, s1;
    seg_bounds<ES>(e0, e1, l, full, s0, s1);
    const DF rem = df_add(r, DF{-excl.hi, -excl.lo});
    return seg_pick<ES>(rs, rt, rd, s0, s1, rem.hi + rem.lo, lane, c_hi, c_lo);
}

// The draw inside chunk [e0, e1) given the remainder r (one warp).  Whole-vector
// chunks: the chunk's 8 round sums (given, or computed here with one coalesced
// pass), a scan over them, then round_pick; other chunks: chunk_pick.
template <int ES>
__device__ int pick_in_chunk(const ReqState& rs, const char* rt, const char* rd, int e0, int e1, DF r,
                             const float* rsum, int lane, float c_hi, float c_lo) {
    if (!chunk_vec<ES>(rs, rt, rd, e0, e1)) return chunk_pick<ES>(rs, rt, rd, e0, e1, r, lane, c_hi, c_lo);
    const int nvec = (e1 - e0) * ES / 16;
    float rv;
    if (rsum) {
        rv = lane < 8 ? rsum[lane] : 0.f;
    } else {
        const float mine = chunk_round_sums<ES>(rs, rt, rd, e0, nvec, lane, c_hi, c_lo);
        rv = __shfl_sync(0xffffffffu, mine, (lane & 7) * 4);
        if (lane >= 8) rv = 0.f;
    }
    DF excl;
    const int k = scan_find(DF{rv, 0.f}, r, lane, excl);
    if (k < 0) return chunk_pick<ES>(rs, rt, rd, e0, e1, DF{INFINITY, 0.f}, lane, c_hi, c_lo);
    const DF rem = df_add(r, DF{-excl.hi, -excl.lo});
    return round_pick<ES>(rs, rt, rd, e0, nvec, k, rem.hi + rem.lo, lane, c_hi, c_lo);
}

// ================================================================== finish
// One thread-block cluster (cs CTAs of 16 warps) per request:
//   1. (before the streaming kernel's results are needed) validation of the
//      request's inputs and the gathers of z at the draft tokens, in every CTA;
//   2. row merges spread over the cluster's warps, each merged row broadcast
//      to every CTA's shared memory (distributed shared memory);
//   3. cluster barrier; every CTA takes the same accept decision (one warp,
//      one ballot); rank 0 writes the accepted prefix;
//   4. T > 0 after a rejection: draw weights summed per chunk and per lane
//      segment across the cluster's warps, written into rank 0's shared memory;
//   5. cluster barrier; rank 0 draws the token by inverse CDF in three scans:
//      chunk totals, the chosen chunk's lane-segment sums, the chosen
//      segment's elements (two-float prefixes).  A bonus draw takes its chunk
//      totals from the streaming kernel's partials and scans the chosen chunk.
struct FinishArgs {
    const char* target;
    const char* draft;
    const int32_t* tokens;
    const int32_t* verify_len;
    const float* uniforms;
    int32_t* out_tokens;
    int32_t* out_accept_len;
    int B, gamma, V;
    float c_hi, c_lo;
    char* ws;
    RowMap rm;
    int stats_grid;  // CTAs of the streaming kernel (one timeout word each)
};

struct RowStatS {
    float M;
    DF S;  // NaN in S.hi marks an invalid row
    int arg;
};

constexpr int kFinWarps = 16;
constexpr int kFinThreads = kFinWarps * 32;
constexpr int kMaxCluster = 4;
constexpr int kChunkSmem = 2048;  // chunk totals kept in rank 0's shared memory
constexpr int kRoundSmem = 1024;  // chunks whose round sums are kept there too

// CTAs per request: enough warps for the rows to merge and the chunks to sum.
inline int finish_cluster_size(int B, int gamma, int nch, bool greedy, int sms) {
    const int rows = greedy ? gamma + 1 : 2 * gamma + 1;
    const int work = greedy ? rows : std::max(rows, nch);
    const int by_work = (work + kFinWarps - 1) / kFinWarps;
    // small batches at T > 0: spread each request's residual sums over more SMs
    const int by_fill = greedy ? 1 : (2 * sms + B - 1) / B;
    return std::min(kMaxCluster, std::max(1, std::max(by_work, by_fill)));
}

// Parts per full-vector chunk in the residual sums: a chunk's 8 rounds are
// split over f warps (8 / f rounds each, one memory round trip) when the
// cluster has at least 2 f warps per chunk.  The same value in both phases.
__host__ __device__ inline int residual_split(int nch, int nw) {
    int f = 1;
    while (f < 8 && nch * f * 2 <= nw) f *= 2;
    return f;
}

// SPLIT: the residual sums are split into (chunk, round group) tasks (small
// vocabularies with warps to spare); a separate instantiation, so that the
// common path's register allocation does not carry that code.
template <int ES, bool GREEDY, bool SPLIT>
__global__ void __launch_bounds__(kFinThreads, 2) k_finish(FinishArgs a, Layout L) {
    cg::cluster_group cluster = cg::this_cluster();
    const int cs = (int)cluster.num_blocks();
    const int rank = (int)cluster.block_rank();
    const int b = blockIdx.x / cs;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gw = rank * kFinWarps + warp, nw = cs * kFinWarps;  // warp within the cluster
    __shared__ RowStatS s_row[2 * SPEC_MAX_GAMMA + 1];
    __shared__ float s_zt[SPEC_MAX_GAMMA], s_zd[SPEC_MAX_GAMMA];
    __shared__ float s_ctot[kChunkSmem];
    __shared__ float s_rsum[kRoundSmem][8];
    __shared__ ReqState s_job;
    __shared__ int s_call_status;
    int* hdr = (int*)(a.ws + L.hdr);
    const float2* partial = (const float2*)(a.ws + L.partial);
    const int G1 = a.gamma + 1, T1 = a.B * G1;
    const int ell = a.verify_len ? a.verify_len[b] : a.gamma;
    // rows_ok: the request's rows exist (the streaming kernel read them)
    const bool ell_ok = ell >= 0 && ell <= a.gamma;
    const bool rows_ok = ell_ok && rows_in_range(a.rm, b, ell, !GREEDY);

    // 1. caller inputs only (ready before the streaming kernel started)
    int st = SPEC_OK;
    int x = 0;
    float uj = 0.f, ug = 0.f, ub = 0.f;
    if (warp == 0) {
        if (!ell_ok) st = SPEC_ERR_VERIFY_LEN;
        else if (!rows_ok) st = SPEC_ERR_ROW_INDEX;
        const int j = lane;
        if (ell_ok && j < ell) x = a.tokens[(size_t)b * a.gamma + j];
        if (!GREEDY && ell_ok) {
            const float* u = a.uniforms + (size_t)b * (a.gamma + 2);
            if (j < ell) uj = u[j];
            ug = u[a.gamma];
            ub = u[a.gamma + 1];
        }
        const bool xok = x >= 0 && x < a.V;
        if (!GREEDY && rows_ok && j < ell) {
            const int xc = xok ? x : 0;
            s_zt[j] = load_logit<ES>(a.target + target_row(a.rm, b, j, G1) * a.V * ES, xc);
            s_zd[j] = load_logit<ES>(a.draft + draft_row(a.rm, b, j, a.gamma) * a.V * ES, xc);
        }
        if (st == SPEC_OK && !__all_sync(0xffffffffu, xok)) st = SPEC_ERR_TOKEN;
        if (st == SPEC_OK && !GREEDY) {
            bool uok = in01(uj);
            if (j == 0) uok = uok && in01(ug) && in01(ub);
            if (!__all_sync(0xffffffffu, uok)) st = SPEC_ERR_UNIFORM;
        }
    }
    pdl_wait();  // the streaming kernel's partials and timeout words
    pdl_trigger();
    // Whether a streaming CTA's wait expired, taken by the cluster's last warp
    // (idle in the merges unless the rows outnumber the warps) and sent to
    // every CTA of the cluster.
    if (gw == nw - 1) {
        const int4* w4 = (const int4*)(a.ws + L.ctaw);
        const int4 v0 = 4 * lane < a.stats_grid ? w4[lane] : make_int4(0, 0, 0, 0);
        const int4 v1 = 4 * (lane + 32) < a.stats_grid ? w4[lane + 32] : make_int4(0, 0, 0, 0);
        const int w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        bool late = false;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int i = (k < 4 ? 4 * lane : 4 * (lane + 32)) + (k & 3);
            late |= i < a.stats_grid && w[k] != SPEC_OK;
        }
        const int v = __any_sync(0xffffffffu, late) ? SPEC_ERR_TIMEOUT : SPEC_OK;
        if (lane < cs) *cluster.map_shared_rank(&s_call_status, lane) = v;
    }

    // 2. row merges: target rows 0..ell, then draft rows 0..ell-1
    const int nrows = rows_ok ? (GREEDY ? ell + 1 : 2 * ell + 1) : 0;
    for (int r = gw; r < nrows; r += nw) {
        const int g = r <= ell ? b * G1 + r : T1 + b * a.gamma + (r - ell - 1);
        RowStatS rs;
        const bool ok = merge_row<GREEDY>(partial + (size_t)g * L.nch, L.nch, lane, rs.M, rs.S, rs.arg);
        if (!ok) rs.S = DF{__int_as_float(0x7fc00000), 0.f};
        if (lane < cs) *cluster.map_shared_rank(&s_row[r], lane) = rs;  // to every CTA of the request
    }
    // a one-CTA cluster (at T = 0) needs only the CTA barrier for its own
    // shared memory; the sampling instantiations keep the cluster barrier only
    if (GREEDY && cs == 1)
        __syncthreads();
    else
        cluster.sync();

    // 3. accept decision (identical in every CTA)
    if (warp == 0) {
        if (s_call_status != SPEC_OK) st = s_call_status;
        if (st == SPEC_OK) {
            bool bad = false;
            for (int r = lane; r < nrows; r += 32) bad |= s_row[r].S.hi != s_row[r].S.hi;
            if (__any_sync(0xffffffffu, bad)) st = SPEC_ERR_NONFINITE;
        }
        int32_t* ot = a.out_tokens + (size_t)b * G1;
        float2* pq = (float2*)(a.ws + L.pq);  // p(x), q(x) diagnostics (fp32; widened by k_copy_stats)
        float2* mass = (float2*)(a.ws + L.mass);
        ReqState o;
        o.ell = ell;
        o.status = st;
        o.n = -1;
        o.mode = 0;
        o.g_t = o.g_d = -1;
        o.u = o.M_t = o.M_d = o.rho_hi = o.rho_lo = 0.f;
        o.S_hi = o.S_lo = 0.f;
        if (st != SPEC_OK) {
            if (rank == 0) {
                for (int k = lane; k <= a.gamma; k += 32) ot[k] = -1;
                for (int k = lane; k < a.gamma; k += 32)
                    pq[(size_t)b * a.gamma + k] = make_float2(__int_as_float(0x7fc00000), __int_as_float(0x7fc00000));
                if (lane == 0) {
                    a.out_accept_len[b] = -1;
                    mass[b] = make_float2(__int_as_float(0x7fc00000), 0.f);
                    set_status(&hdr[kHdrStatus], st);
                }
            }
        } else {
            // accept tests, one lane per position (gamma <= 32): u * q(x) < p(x)
            const int j = lane;
            bool acc = true;
            float px = __int_as_float(0x7fc00000), qx = px;
            DF rho_j = {0.f, 0.f};  // S_t / S_d of position j, in case the draw is its residual
            if (j < ell) {
                if (GREEDY) {
                    acc = x == s_row[j].arg;
                } else {
                    px = div_df(scaled_exp(s_zt[j], a.c_hi, a.c_lo, s_row[j].M), s_row[j].S);
                    qx = div_df(scaled_exp(s_zd[j], a.c_hi, a.c_lo, s_row[ell + 1 + j].M), s_row[ell + 1 + j].S);
                    acc = __fmul_rn(uj, qx) < px;
                    rho_j = df_div(s_row[j].S, s_row[ell + 1 + j].S);
                }
            }
            const unsigned rej = __ballot_sync(0xffffffffu, !acc);
            const int n = rej ? min(__ffs(rej) - 1, ell) : ell;
            const DF St = s_row[n].S;
            o.n = n;
            o.g_t = b * G1 + n;
            o.M_t = s_row[n].M;
            o.S_hi = St.hi;
            o.S_lo = St.lo;
            const float rho_hi = __shfl_sync(0xffffffffu, rho_j.hi, n & 31);
            const float rho_lo = __shfl_sync(0xffffffffu, rho_j.lo, n & 31);
            if (!GREEDY && n < ell) {
                o.mode = 1;
                o.g_d = T1 + b * a.gamma + n;
                o.M_d = s_row[ell + 1 + n].M;
                o.rho_hi = rho_hi;
                o.rho_lo = rho_lo;
                o.u = ug;
            } else if (!GREEDY) {
                o.mode = 2;
                o.u = ub;
            }
            if (rank == 0) {
                if (j < a.gamma) pq[(size_t)b * a.gamma + j] = make_float2(px, qx);
                // lane k holds draft token k; slot gamma (32 at most) needs lane 0's help
                if (lane < n) ot[lane] = x;
                else if (lane > n && lane <= a.gamma) ot[lane] = -1;
                if (lane == 0 && a.gamma == 32 && n < 32) ot[32] = -1;
                if (lane == 0) {
                    a.out_accept_len[b] = n;
                    mass[b] = make_float2(__int_as_float(0x7fc00000), 0.f);
                    if (GREEDY) ot[n] = s_row[n].arg;
                }
            }
        }
        if (lane == 0) {
            s_job = o;
            if (rank == 0) ((ReqState*)(a.ws + L.req))[b] = o;
        }
    }
    __syncthreads();
    if (GREEDY) return;
    ReqState job = s_job;
    if (job.status != SPEC_OK) return;  // the same in every CTA of the cluster

    // 4. residual sums per chunk and per lane segment over the cluster's warps
    const char* rt = a.target + target_row(a.rm, b, job.n, G1) * a.V * ES;
    const char* rd = job.mode == 1 ? a.draft + draft_row(a.rm, b, job.n, a.gamma) * a.V * ES : rt;
    float* rchunk = (float*)(a.ws + L.rchunk) + (size_t)b * L.nch;
    const bool tot_smem = L.nch <= kChunkSmem;
    const bool round_smem = L.nch <= kRoundSmem;
    const int fsplit = SPLIT && round_smem ? residual_split(L.nch, nw) : 1;
    if (SPLIT && job.mode == 1 && fsplit > 1) {
        // (chunk, round group) tasks; chunk totals are summed from the round
        // sums by rank 0 before the draw
        const int R = 8 / fsplit;
        for (int task = gw; task < L.nch * fsplit; task += nw) {
            const int c = task / fsplit, part = task - c * fsplit;
            const int e0 = c * L.CH, e1 = min(a.V, e0 + L.CH);
            if (chunk_vec<ES>(job, rt, rd, e0, e1)) {
                const int nvec = (e1 - e0) * ES / 16;
                const uint4* vt = (const uint4*)(rt + (size_t)e0 * ES);
                const uint4* vd = (const uint4*)(rd + (size_t)e0 * ES);
                uint4 tv[4], dv[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int i = 32 * (part * R + k) + lane;
                    tv[k] = dv[k] = make_uint4(0, 0, 0, 0);
                    if (k < R && i < nvec) {
                        tv[k] = __ldg(vt + i);
                        dv[k] = __ldg(vd + i);
                    }
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    if (k < R) {
                        const int i = 32 * (part * R + k) + lane;
                        const float w = i < nvec ? vec_weight_sum_ordered<ES>(job, tv[k], dv[k], a.c_hi, a.c_lo) : 0.f;
                        const float rsum = warp_sum(w);
                        if (lane == 0) *cluster.map_shared_rank(&s_rsum[c][part * R + k], 0) = rsum;
                    }
                }
            } else if (part == 0) {
                int lpos;
                const float ls = seg_weight_sum<ES>(job, rt, rd, e0, e1, false, lane, a.c_hi, a.c_lo, lpos);
                const DF tot = warp_sum_df(DF{ls, 0.f});
                if (lane == 0) *cluster.map_shared_rank(&s_ctot[c], 0) = tot.hi + tot.lo;
            }
        }
    } else if (!SPLIT && job.mode == 1) {
        for (int c = gw; c < L.nch; c += nw) {
            const int e0 = c * L.CH, e1 = min(a.V, e0 + L.CH);
            float t;
            if (chunk_vec<ES>(job, rt, rd, e0, e1)) {
                // lane l holds the total of round l >> 2
                const float rsum =
                    chunk_round_sums<ES>(job, rt, rd, e0, (e1 - e0) * ES / 16, lane, a.c_hi, a.c_lo);
                if (round_smem && (lane & 3) == 0) *cluster.map_shared_rank(&s_rsum[c][lane >> 2], 0) = rsum;
                DF acc = {0.f, 0.f};
#pragma unroll
                for (int k = 0; k < 8; ++k) acc = df_add(acc, DF{__shfl_sync(0xffffffffu, rsum, 4 * k), 0.f});
                t = acc.hi + acc.lo;
            } else {
                int lpos;
                const float ls = seg_weight_sum<ES>(job, rt, rd, e0, e1, false, lane, a.c_hi, a.c_lo, lpos);
                const DF tot = warp_sum_df(DF{ls, 0.f});
                t = tot.hi + tot.lo;
            }
            if (lane == 0) {
                if (tot_smem) *cluster.map_shared_rank(&s_ctot[c], 0) = t;
                else rchunk[c] = t;
            }
        }
        if (!tot_smem) __threadfence();
    }
    cluster.sync();
    if (rank != 0 || warp != 0) return;

    // 5. the draw (rank 0, warp 0); the request's state is read from shared
    // memory here, so that the draw fits in the register budget without spills
    ReqState& jd = s_job;
    if (SPLIT && jd.mode == 1 && fsplit > 1) {
        // totals of the split chunks from their round sums, in round order
        for (int c = lane; c < L.nch; c += 32) {
            const int e0 = c * L.CH, e1 = min(a.V, e0 + L.CH);
            if (chunk_vec<ES>(jd, rt, rd, e0, e1)) {
                DF acc = {0.f, 0.f};
#pragma unroll
                for (int k = 0; k < 8; ++k) acc = df_add(acc, DF{s_rsum[c][k], 0.f});
                s_ctot[c] = acc.hi + acc.lo;
            }
        }
        __syncwarp();
    }
    const float2* tpart = partial + (size_t)jd.g_t * L.nch;
    auto total_of = [&](const ReqState& js, int c) -> float {
        if (js.mode == 1) return tot_smem ? s_ctot[c] : __ldcg(rchunk + c);
        const float2 p = tpart[c];
        if (p.x == -INFINITY) return 0.f;
        const float d = p.x - js.M_t;
        return p.y * pow2_f(d < -1000.f ? -1000 : (int)d);
    };
    // Chunk totals, each lane taking a block of consecutive chunks: the lane
    // sums (in chunk order) and one inclusive two-float warp scan of them give
    // the total W (lane 31) and the lane whose block the draw falls in; that
    // lane walks its block from its exclusive prefix.
    const int cpl = (L.nch + 31) / 32;
    const int k0 = min(L.nch, lane * cpl), k1 = min(L.nch, k0 + cpl);
    DF lsum, incl;
    int lpos;  // this lane's last chunk with positive total, or -1
    auto block_scan = [&]() {
        lsum = DF{0.f, 0.f};
        lpos = -1;
#pragma unroll 4
        for (int k = k0; k < k1; ++k) {
            const float v = total_of(jd, k);
            lsum = df_add(lsum, DF{v, 0.f});
            if (v > 0.f) lpos = k;
        }
        incl = warp_scan_df(lsum, lane);
    };
    block_scan();
    DF W = {__shfl_sync(0xffffffffu, incl.hi, 31), __shfl_sync(0xffffffffu, incl.lo, 31)};
    if (!(W.hi > 0.f) && jd.mode == 1) {
        // the residual summed to zero: draw from p of the same row instead
        jd.mode = 2;
        rd = rt;
        if (lane == 0) atomicOr(&hdr[kHdrEvents], 1);
        block_scan();
        W = DF{__shfl_sync(0xffffffffu, incl.hi, 31), __shfl_sync(0xffffffffu, incl.lo, 31)};
    }
    // target = u * W as a two-float number
    DF target;
    {
        const float p = jd.u * W.hi;
        const float pe = fmaf(jd.u, W.hi, -p);
        target = df_add(DF{p, 0.f}, DF{pe + jd.u * W.lo, 0.f});
    }
    auto exceeds = [](DF x, DF t) { return x.hi > t.hi || (x.hi == t.hi && x.lo > t.lo); };
    int cstar = -1;
    DF before = {0.f, 0.f};
    const unsigned hit = __ballot_sync(0xffffffffu, exceeds(incl, target));
    if (hit) {
        const int l = __ffs(hit) - 1;
        DF excl = {__shfl_up_sync(0xffffffffu, incl.hi, 1), __shfl_up_sync(0xffffffffu, incl.lo, 1)};
        if (lane == 0) excl = DF{0.f, 0.f};
        if (lane == l) {
            // the first chunk whose running prefix exceeds the target; if
            // rounding of the walk leaves none, the block's last chunk with
            // positive weight (the draw's rule for a target at the very end)
            DF run = excl;
            int lastp = -1;
            DF before_lastp = excl;
            for (int k = k0; k < k1; ++k) {
                const float v = total_of(jd, k);
                const DF next = df_add(run, DF{v, 0.f});
                if (v > 0.f) {
                    lastp = k;
                    before_lastp = run;
                }
                if (exceeds(next, target)) {
                    cstar = k;
                    before = run;
                    break;
                }
                run = next;
            }
            if (cstar < 0) {
                cstar = lastp >= 0 ? lastp : k1 - 1;
                before = lastp >= 0 ? before_lastp : run;
            }
        }
        cstar = __shfl_sync(0xffffffffu, cstar, l);
        before.hi = __shfl_sync(0xffffffffu, before.hi, l);
        before.lo = __shfl_sync(0xffffffffu, before.lo, l);
    }
    int last_pos = lpos;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) last_pos = max(last_pos, __shfl_xor_sync(0xffffffffu, last_pos, o));
    int tok;
    if (cstar < 0) {
        // rounding left no chunk: the last element with positive weight of the
        // last chunk with positive weight
        cstar = last_pos >= 0 ? last_pos : L.nch - 1;
        const int e0 = cstar * L.CH, e1 = min(a.V, e0 + L.CH);
        tok = chunk_pick<ES>(jd, rt, rd, e0, e1, DF{INFINITY, 0.f}, lane, a.c_hi, a.c_lo);
        if (lane == 0) atomicOr(&hdr[kHdrEvents], 2);
    } else {
        const DF r = df_add(target, DF{-before.hi, -before.lo});
        const int e0 = cstar * L.CH, e1 = min(a.V, e0 + L.CH);
        const float* rsum = (jd.mode == 1 && round_smem) ? s_rsum[cstar] : nullptr;
        tok = pick_in_chunk<ES>(jd, rt, rd, e0, e1, r, rsum, lane, a.c_hi, a.c_lo);
    }
    if (lane == 0) {
        a.out_tokens[(size_t)b * G1 + jd.n] = tok;
        ((float2*)(a.ws + L.mass))[b] = make_float2(W.hi, W.lo);  // divided by S_t in k_copy_stats
    }
}

// ==================================================================== stats
__global__ void k_copy_stats(const char* ws, Layout L, int B, int gamma, double* px, double* qx,
                             double* mass, int32_t* status) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    const float2* pq = (const float2*)(ws + L.pq);
    if (i < B * gamma) {
        if (px) px[i] = (double)pq[i].x;
        if (qx) qx[i] = (double)pq[i].y;
    }
    if (i < B) {
        const ReqState rs = ((const ReqState*)(ws + L.req))[i];
        const float2 w = ((const float2*)(ws + L.mass))[i];
        // the draw's total weight over the target row sum, both float pairs
        if (mass)
            mass[i] = rs.status == SPEC_OK
                          ? ((double)w.x + (double)w.y) / ((double)rs.S_hi + (double)rs.S_lo)
                          : __longlong_as_double(0x7ff8000000000000ll);
        if (status) status[i] = rs.status;
    }
}

// Dense request-major packing of the rows of ragged prefixes: exclusive
// prefix sums of ell_b + 1 (target rows) and ell_b (draft rows).  One CTA.
constexpr int kPackThreads = 1024;

__global__ void __launch_bounds__(kPackThreads) k_pack_rows(const int32_t* verify_len, int B, int gamma,
                                                            int32_t* trow, int32_t* drow, int32_t* totals) {
    __shared__ int s_t[32], s_d[32];
    pdl_trigger();  // the verification that follows may be placed now (it waits for these results)
    constexpr int PER = (SPEC_MAX_BATCH + kPackThreads - 1) / kPackThreads;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int ct[PER], cd[PER], mt = 0, md = 0;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int b = tid * PER + i;
        const int ell = b < B ? verify_len[b] : -1;
        const bool ok = ell >= 0 && ell <= gamma;
        ct[i] = ok ? ell + 1 : 0;
        cd[i] = ok ? ell : 0;
        mt += ct[i];
        md += cd[i];
    }
    int it = mt, id = md;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int vt = __shfl_up_sync(0xffffffffu, it, o), vd = __shfl_up_sync(0xffffffffu, id, o);
        if (lane >= o) {
            it += vt;
            id += vd;
        }
    }
    if (lane == 31) {
        s_t[warp] = it;
        s_d[warp] = id;
    }
    __syncthreads();
    if (warp == 0) {
        const int wt = s_t[lane], wd = s_d[lane];
        int xt = wt, xd = wd;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int vt = __shfl_up_sync(0xffffffffu, xt, o), vd = __shfl_up_sync(0xffffffffu, xd, o);
            if (lane >= o) {
                xt += vt;
                xd += vd;
            }
        }
        s_t[lane] = xt - wt;
        s_d[lane] = xd - wd;
        if (lane == 31) {
            totals[0] = xt;
            totals[1] = xd;
        }
    }
    __syncthreads();
    int ot = s_t[warp] + it - mt, od = s_d[warp] + id - md;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int b = tid * PER + i;
        if (b < B) {
            trow[b] = ot;
            drow[b] = od;
        }
        ot += ct[i];
        od += cd[i];
    }
}

}  // namespace specv

// ===================================================================== host
using namespace specv;

namespace {

// profiling hook (spec_profile_events): atomics, so that setting it from one
// thread while another launches is not a data race
std::atomic<cudaEvent_t> g_ev_before{nullptr}, g_ev_after{nullptr};
// test hook (spec_selftest_expire_first_wait)
std::atomic<int> g_expire_first{0};

struct DeviceInfo {
    int sms = 0;
    bool attrs_set = false;
};
std::mutex g_mu;
DeviceInfo g_dev[64];

int device_info(int& sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SPEC_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.attrs_set) {
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return SPEC_ERR_CUDA;
        const void* fns[16] = {
            (const void*)k_row_stats<2, false, false, false>, (const void*)k_row_stats<2, true, false, false>,
            (const void*)k_row_stats<4, false, false, false>, (const void*)k_row_stats<4, true, false, false>,
            (const void*)k_row_stats<2, false, true, false>,  (const void*)k_row_stats<2, true, true, false>,
            (const void*)k_row_stats<4, false, true, false>,  (const void*)k_row_stats<4, true, true, false>,
            (const void*)k_row_stats<2, false, false, true>,  (const void*)k_row_stats<2, true, false, true>,
            (const void*)k_row_stats<4, false, false, true>,  (const void*)k_row_stats<4, true, false, true>,
            (const void*)k_row_stats<2, false, true, true>,   (const void*)k_row_stats<2, true, true, true>,
            (const void*)k_row_stats<4, false, true, true>,   (const void*)k_row_stats<4, true, true, true>};
        for (int i = 0; i < 16; ++i)  // entries 8..15: the packed layout's instantiations
            if (cudaFuncSetAttribute(fns[i], cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)(i < 8 ? kStatsSmem : kStatsSmemPacked)) != cudaSuccess)
                return SPEC_ERR_CUDA;
        d.attrs_set = true;
    }
    sms = d.sms;
    return SPEC_OK;
}

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

int check_shape(int B, int gamma, int V, spec_dtype dt) {
    if (B < 0 || B > SPEC_MAX_BATCH || gamma < 0 || gamma > SPEC_MAX_GAMMA || V < 1) return SPEC_ERR_SHAPE;
    if (dt != SPEC_F32 && dt != SPEC_BF16) return SPEC_ERR_SHAPE;
    return SPEC_OK;
}

template <int ES, bool GREEDY>
int launch_chain(const StatsArgs& sa, const FinishArgs& fa, const Layout& L, int sms, bool aligned_rows,
                 cudaStream_t st) {
    const long long max_items = (long long)L.R * L.nch;
    const int grid = (int)std::min<long long>(std::min(sms, kMaxStatsGrid), (max_items + kStatsWarps - 1) / kStatsWarps);
    const bool packed = sa.rm.trow != nullptr;
    const cudaEvent_t ev_before = g_ev_before.load(std::memory_order_relaxed);
    const cudaEvent_t ev_after = g_ev_after.load(std::memory_order_relaxed);
    if (ev_before) cudaEventRecord(ev_before, st);
    {
        // a programmatic dependent of the preceding kernel (the previous call's
        // finish kernel, say): its CTAs are placed as that kernel drains and
        // wait in griddepcontrol.wait instead of being launched after it
        cudaLaunchAttribute pa[1];
        pa[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        pa[0].val.programmaticStreamSerializationAllowed = 1;
        cudaLaunchConfig_t kc = {};
        kc.gridDim = dim3((unsigned)grid);
        kc.blockDim = dim3(kStatsThreads);
        kc.dynamicSmemBytes = packed ? kStatsSmemPacked : kStatsSmem;
        kc.stream = st;
        kc.attrs = pa;
        kc.numAttrs = 1;
        cudaError_t ke;
        if (aligned_rows) ke = packed ? cudaLaunchKernelEx(&kc, k_row_stats<ES, GREEDY, true, true>, sa, L)
                                      : cudaLaunchKernelEx(&kc, k_row_stats<ES, GREEDY, true, false>, sa, L);
        else ke = packed ? cudaLaunchKernelEx(&kc, k_row_stats<ES, GREEDY, false, true>, sa, L)
                         : cudaLaunchKernelEx(&kc, k_row_stats<ES, GREEDY, false, false>, sa, L);
        if (ke != cudaSuccess) return SPEC_ERR_CUDA;
    }
    if (ev_after) cudaEventRecord(ev_after, st);
    FinishArgs fa2 = fa;
    fa2.stats_grid = grid;
    // one cluster per request; it may be scheduled while the streaming kernel
    // finishes and waits for its results with griddepcontrol.wait
    const int cs = finish_cluster_size(sa.B, sa.gamma, L.nch, GREEDY, sms);
    const bool split = !GREEDY && L.nch <= kRoundSmem && residual_split(L.nch, cs * kFinWarps) > 1;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)cs;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(sa.B * cs));
    cfg.blockDim = dim3(kFinThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e;
    if (GREEDY || !split) e = cudaLaunchKernelEx(&cfg, k_finish<ES, GREEDY, false>, fa2, L);
    else e = cudaLaunchKernelEx(&cfg, k_finish<ES, GREEDY, !GREEDY>, fa2, L);
    if (e != cudaSuccess) return SPEC_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

int verify_impl(const void* target_logits, const void* draft_logits, const RowMap& rm, spec_dtype dt, int B,
                int gamma, int V, const int32_t* draft_tokens, const int32_t* verify_len, float temperature,
                const float* uniforms, int32_t* out_tokens, int32_t* out_accept_len, void* workspace,
                size_t workspace_bytes, spec_stream_t stream) {
    int rc = check_shape(B, gamma, V, dt);
    if (rc != SPEC_OK) return rc;
    if (!(temperature == 0.0f || (temperature >= 1e-4f && temperature <= 1e4f)))
        return SPEC_ERR_TEMPERATURE;
    if (B == 0) return SPEC_OK;
    const bool greedy = temperature == 0.0f;
    const int es = dt == SPEC_BF16 ? 2 : 4;
    if (!target_logits || !out_tokens || !out_accept_len || !workspace) return SPEC_ERR_NULL;
    if (gamma > 0 && !draft_tokens) return SPEC_ERR_NULL;
    if (!greedy && gamma > 0 && !draft_logits) return SPEC_ERR_NULL;
    if (!greedy && !uniforms) return SPEC_ERR_NULL;
    if (!aligned(target_logits, es) || (draft_logits && !aligned(draft_logits, es)) ||
        (draft_tokens && !aligned(draft_tokens, 4)) || (verify_len && !aligned(verify_len, 4)) ||
        (uniforms && !aligned(uniforms, 4)) || !aligned(out_tokens, 4) || !aligned(out_accept_len, 4) ||
        !aligned(workspace, 16))
        return SPEC_ERR_ALIGN;
    const Layout L(B, gamma, V, es);
    if (workspace_bytes < L.total) return SPEC_ERR_WORKSPACE;
    int sms = 0;
    rc = device_info(sms);
    if (rc != SPEC_OK) return rc;

    // scale c = log2(e) / T as an unevaluated pair c_hi + c_lo with c_lo > 0
    const double c = greedy ? 1.0 : 1.4426950408889634074 / (double)temperature;
    float c_hi = (float)c;
    if ((double)c_hi >= c) c_hi = nextafterf(c_hi, 0.0f);
    const float c_lo = (float)(c - (double)c_hi);

    const char* t = (const char*)target_logits;
    const char* d = (const char*)draft_logits;
    char* ws = (char*)workspace;
    StatsArgs sa{t, d, verify_len, B, gamma, V, c_hi, c_lo, ws, rm, g_expire_first.load(std::memory_order_relaxed)};
    FinishArgs fa{t,    d,    draft_tokens, verify_len, uniforms, out_tokens, out_accept_len, B, gamma, V,
                  c_hi, c_lo, ws,           rm,         0};
    cudaStream_t st = (cudaStream_t)stream;
    // every row starts on a 16-byte boundary: whole-chunk copies
    const bool al = aligned(target_logits, 16) && (greedy || gamma == 0 || !draft_logits || aligned(draft_logits, 16)) &&
                    ((size_t)V * es) % 16 == 0;
    if (es == 2)
        return greedy ? launch_chain<2, true>(sa, fa, L, sms, al, st) : launch_chain<2, false>(sa, fa, L, sms, al, st);
    return greedy ? launch_chain<4, true>(sa, fa, L, sms, al, st) : launch_chain<4, false>(sa, fa, L, sms, al, st);
}

}  // namespace

extern "C" {

size_t spec_verify_workspace_bytes(int B, int gamma, int V, spec_dtype dt) {
    if (check_shape(B, gamma, V, dt) != SPEC_OK) return 0;
    return Layout(B, gamma, V, dt == SPEC_BF16 ? 2 : 4).total;
}

int spec_verify(const void* target_logits, const void* draft_logits, spec_dtype dt, int B, int gamma,
                int V, const int32_t* draft_tokens, const int32_t* verify_len, float temperature,
                const float* uniforms, int32_t* out_tokens, int32_t* out_accept_len, void* workspace,
                size_t workspace_bytes, spec_stream_t stream) {
    TraceRange tr("spec_verify");
    return verify_impl(target_logits, draft_logits, RowMap{nullptr, nullptr, 0, 0}, dt, B, gamma, V, draft_tokens,
                       verify_len, temperature, uniforms, out_tokens, out_accept_len, workspace, workspace_bytes,
                       stream);
}

int spec_verify_packed(const void* target_logits, int K_target, const void* draft_logits, int K_draft,
                       const int32_t* target_row, const int32_t* draft_row, spec_dtype dt, int B, int gamma, int V,
                       const int32_t* draft_tokens, const int32_t* verify_len, float temperature,
                       const float* uniforms, int32_t* out_tokens, int32_t* out_accept_len, void* workspace,
                       size_t workspace_bytes, spec_stream_t stream) {
    TraceRange tr("spec_verify_packed");
    if (K_target < 0 || K_draft < 0) return SPEC_ERR_SHAPE;
    if (B > 0) {
        if (!target_row) return SPEC_ERR_NULL;
        if (temperature != 0.0f && gamma > 0 && !draft_row) return SPEC_ERR_NULL;
        if (!aligned(target_row, 4) || (draft_row && !aligned(draft_row, 4))) return SPEC_ERR_ALIGN;
    }
    return verify_impl(target_logits, draft_logits, RowMap{target_row, draft_row, K_target, K_draft}, dt, B, gamma,
                       V, draft_tokens, verify_len, temperature, uniforms, out_tokens, out_accept_len, workspace,
                       workspace_bytes, stream);
}

int spec_pack_rows(const int32_t* verify_len, int B, int gamma, int32_t* target_row, int32_t* draft_row,
                   int32_t* totals, spec_stream_t stream) {
    TraceRange tr("spec_pack_rows");
    if (B < 0 || B > SPEC_MAX_BATCH || gamma < 0 || gamma > SPEC_MAX_GAMMA) return SPEC_ERR_SHAPE;
    if (!totals) return SPEC_ERR_NULL;
    if (B > 0 && (!verify_len || !target_row || !draft_row)) return SPEC_ERR_NULL;
    if (!aligned(totals, 4) || (verify_len && !aligned(verify_len, 4)) || (target_row && !aligned(target_row, 4)) ||
        (draft_row && !aligned(draft_row, 4)))
        return SPEC_ERR_ALIGN;
    k_pack_rows<<<1, kPackThreads, 0, (cudaStream_t)stream>>>(verify_len, B, gamma, target_row, draft_row, totals);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

int spec_verify_stats(const void* workspace, size_t workspace_bytes, int B, int gamma, int V,
                      spec_dtype dt, double* px, double* qx, double* resid_mass, int32_t* status,
                      spec_stream_t stream) {
    const int rc = check_shape(B, gamma, V, dt);
    if (rc != SPEC_OK) return rc;
    if (B == 0) return SPEC_OK;
    if (!workspace) return SPEC_ERR_NULL;
    const Layout L(B, gamma, V, dt == SPEC_BF16 ? 2 : 4);
    if (workspace_bytes < L.total) return SPEC_ERR_WORKSPACE;
    const int n = std::max(B * gamma, B);
    k_copy_stats<<<(n + 255) / 256, 256, 0, (cudaStream_t)stream>>>((const char*)workspace, L, B, gamma,
                                                                    px, qx, resid_mass, status);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

int spec_profile_events(void* before_row_stats, void* after_row_stats) {
    g_ev_before.store((cudaEvent_t)before_row_stats, std::memory_order_relaxed);
    g_ev_after.store((cudaEvent_t)after_row_stats, std::memory_order_relaxed);
    return SPEC_OK;
}

int spec_selftest_expire_first_wait(int on) {
    g_expire_first.store(on ? 1 : 0, std::memory_order_relaxed);
    return SPEC_OK;
}

int spec_verify_kernel_count(int B, float temperature) {
    if (B <= 0) return 0;
    return 2;
}

}  // extern "C"
