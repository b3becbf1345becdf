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
// Kernel chain on the caller's stream (no host synchronisation):
//   k_row_stats  persistent, one CTA per SM: the HBM pass.  Each CTA first
//                derives the needed rows from verify_len (target 0..ell, draft
//                0..ell-1).  Each warp then streams 4 KiB row chunks through its
//                own ring of shared-memory stages filled by 1-D bulk copies
//                (cp.async.bulk + mbarrier) and writes one partial per chunk:
//                (integer scale, sum of 2^(z*c - scale)) or (max, argmax).
//   k_accept     one CTA per request: validates the request, merges chunk
//                partials per row (exact power-of-two rescaling, fp64 sums),
//                computes p(x), q(x), runs the accept tests with one warp
//                ballot, writes the accepted prefix and the draw job.
//   k_draw       one warp per (request, chunk) (T > 0): weights of the 1-2
//                draw rows summed per chunk; the warp finishing a request's
//                last chunk takes the fp64 prefix over chunks and scans the
//                chosen chunk for the inverse-CDF draw.
#include <math.h>

#include <algorithm>
#include <mutex>

#include "specv_rowstats.cuh"

namespace specv {

constexpr int kReqThreads = 512;  // accept / draw kernels

__device__ __forceinline__ bool in01(float u) { return u >= 0.0f && u < 1.0f; }

// =================================================================== accept
struct AcceptArgs {
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
};

// Merge the chunk partials of one row.  T > 0: M = max of the chunks'
// integer scales, S = sum_c S_c * 2^(M_c - M) with exact power-of-two rescaling
// and a two-float accumulator.  T == 0: (max, lowest argmax).  Returns false
// for an invalid row.
template <bool GREEDY>
__device__ __forceinline__ bool merge_row(const float2* part, int nch, int lane, float& M, DF& S, int& arg) {
    if (GREEDY) {
        float best = -INFINITY;
        int ix = 0x7fffffff;
        bool bad = false;
        for (int c = lane; c < nch; c += 32) {
            const float2 p = part[c];
            const int i = __float_as_int(p.y);
            if (p.x != p.x) bad = true;
            else if (p.x > best || (p.x == best && i < ix)) { best = p.x; ix = i; }
        }
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
    float2 keep[4];
    int nk = 0;
    for (int c = lane; c < nch; c += 32) {
        const float2 p = part[c];
        if (nk < 4) keep[nk++] = p;
        m = fmax_nan(m, p.x);
    }
    m = warp_max_nan(m);
    M = m;
    arg = 0;
    if (m != m || m == -INFINITY) return false;
    DF acc = {0.f, 0.f};
    int k = 0;
    for (int c = lane; c < nch; c += 32, ++k) {
        const float2 p = k < 4 ? keep[k] : part[c];
        if (p.x != -INFINITY) {
            // both scales are integer-valued: the rescale is an exact power of two
            const float d = p.x - m;
            const float v = p.y * pow2_f(d < -1000.f ? -1000 : (int)d);
            acc = df_add(acc, DF{v, 0.f});
        }
    }
    S = warp_sum_df(acc);
    return S.hi > 0.f && S.hi <= 3.0e38f;
}

// p = e / (S.hi + S.lo) in fp32
__device__ __forceinline__ float div_df(float e, DF S) {
    const float q = e / S.hi;
    return fmaf(-q, S.lo / S.hi, q);
}

template <int ES, bool GREEDY>
__global__ void __launch_bounds__(kReqThreads) k_accept(AcceptArgs a, Layout L) {
    constexpr int NW = kReqThreads / 32;
    const int b = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    __shared__ float s_M[2 * SPEC_MAX_GAMMA + 1];
    __shared__ DF s_S[2 * SPEC_MAX_GAMMA + 1];
    __shared__ int s_arg[2 * SPEC_MAX_GAMMA + 1];
    __shared__ float s_zt[SPEC_MAX_GAMMA], s_zd[SPEC_MAX_GAMMA];
    __shared__ int s_status;
    int* hdr = (int*)(a.ws + L.hdr);
    ReqState* req = (ReqState*)(a.ws + L.req);
    const float2* partial = (const float2*)(a.ws + L.partial);
    double* pq = (double*)(a.ws + L.pq);
    const int G1 = a.gamma + 1, T1 = a.B * G1;
    const int ell = a.verify_len ? a.verify_len[b] : a.gamma;
    const bool ell_ok = ell >= 0 && ell <= a.gamma;

    int st = SPEC_OK;
    if (warp == 0) {
        // caller inputs only (ready before the streaming kernel started):
        // validation and the gathers of z at the (clamped) draft tokens
        if (!ell_ok) st = SPEC_ERR_VERIFY_LEN;
        const int j = lane;
        int x = 0;
        float uj = 0.f, ug = 0.f, ub = 0.f;
        if (ell_ok && j < ell) x = a.tokens[(size_t)b * a.gamma + j];
        if (!GREEDY && ell_ok) {
            const float* u = a.uniforms + (size_t)b * (a.gamma + 2);
            if (j < ell) uj = u[j];
            if (j == 0) {
                ug = u[a.gamma];
                ub = u[a.gamma + 1];
            }
        }
        const bool xok = x >= 0 && x < a.V;
        if (!GREEDY && ell_ok && j < ell) {
            const int xc = xok ? x : 0;
            s_zt[j] = load_logit<ES>(a.target + (size_t)(b * G1 + j) * a.V * ES, xc);
            s_zd[j] = load_logit<ES>(a.draft + (size_t)(b * a.gamma + j) * a.V * ES, xc);
        }
        if (st == SPEC_OK && !__all_sync(0xffffffffu, xok)) st = SPEC_ERR_TOKEN;
        if (st == SPEC_OK && !GREEDY) {
            bool uok = in01(uj);
            if (j == 0) uok = uok && in01(ug) && in01(ub);
            if (!__all_sync(0xffffffffu, uok)) st = SPEC_ERR_UNIFORM;
        }
    }
    pdl_wait();  // the streaming kernel's partials and status word
    pdl_trigger();
    if (warp == 0) {
        if (hdr[kHdrStatus] == SPEC_ERR_TIMEOUT) st = SPEC_ERR_TIMEOUT;
        if (lane == 0) {
            s_status = st;
            ((int*)(a.ws + L.ticket))[b] = 0;  // completion ticket of the draw kernel
        }
    } else if (ell_ok) {
        // row merges: target rows 0..ell, then draft rows 0..ell-1
        const int nrows = GREEDY ? ell + 1 : 2 * ell + 1;
        for (int r = warp - 1; r < nrows; r += NW - 1) {
            const int g = r <= ell ? b * G1 + r : T1 + b * a.gamma + (r - ell - 1);
            float M;
            DF S;
            int arg;
            const bool ok = merge_row<GREEDY>(partial + (size_t)g * L.nch, L.nch, lane, M, S, arg);
            if (lane == 0) {
                s_M[r] = M;
                s_S[r] = ok ? S : DF{__int_as_float(0x7fc00000), 0.f};  // NaN marks an invalid row
                s_arg[r] = arg;
            }
        }
    }
    __syncthreads();
    if (warp != 0) return;

    st = s_status;
    if (st == SPEC_OK) {
        const int nrows = GREEDY ? ell + 1 : 2 * ell + 1;
        bool bad = false;
        for (int r = lane; r < nrows; r += 32) bad |= s_S[r].hi != s_S[r].hi;
        if (__any_sync(0xffffffffu, bad)) st = SPEC_ERR_NONFINITE;
    }
    int32_t* ot = a.out_tokens + (size_t)b * G1;
    const int j = lane;
    if (st != SPEC_OK) {
        for (int k = lane; k <= a.gamma; k += 32) ot[k] = -1;
        for (int k = lane; k < a.gamma; k += 32) {
            pq[2 * ((size_t)b * a.gamma + k)] = __longlong_as_double(0x7ff8000000000000ll);
            pq[2 * ((size_t)b * a.gamma + k) + 1] = __longlong_as_double(0x7ff8000000000000ll);
        }
        if (lane == 0) {
            a.out_accept_len[b] = -1;
            ReqState o;
            o.ell = 0;
            o.status = st;
            o.n = -1;
            o.mode = 0;
            req[b] = o;
            ((double*)(a.ws + L.mass))[b] = __longlong_as_double(0x7ff8000000000000ll);
            set_status(&hdr[kHdrStatus], st);
        }
        return;
    }

    // accept tests, one lane per position (gamma <= 32): u * q(x) < p(x)
    const int32_t* x = a.tokens + (size_t)b * a.gamma;
    bool acc = true;
    double pxd = __longlong_as_double(0x7ff8000000000000ll), qxd = pxd;
    if (j < ell) {
        if (GREEDY) {
            acc = x[j] == s_arg[j];
        } else {
            const float px = div_df(scaled_exp(s_zt[j], a.c_hi, a.c_lo, s_M[j]), s_S[j]);
            const float qx = div_df(scaled_exp(s_zd[j], a.c_hi, a.c_lo, s_M[ell + 1 + j]), s_S[ell + 1 + j]);
            const float u = a.uniforms[(size_t)b * (a.gamma + 2) + j];
            acc = __fmul_rn(u, qx) < px;
            pxd = px;
            qxd = qx;
        }
    }
    if (j < a.gamma) {
        pq[2 * ((size_t)b * a.gamma + j)] = pxd;
        pq[2 * ((size_t)b * a.gamma + j) + 1] = qxd;
    }
    const unsigned rej = __ballot_sync(0xffffffffu, !acc);
    const int n = rej ? min(__ffs(rej) - 1, ell) : ell;
    for (int k = lane; k <= a.gamma; k += 32) {
        if (k < n) ot[k] = x[k];
        else if (k > n) ot[k] = -1;
    }
    if (lane == 0) {
        a.out_accept_len[b] = n;
        ((double*)(a.ws + L.mass))[b] = __longlong_as_double(0x7ff8000000000000ll);
        ReqState o;
        o.ell = ell;
        o.status = SPEC_OK;
        o.n = n;
        o.mode = 0;
        o.g_t = b * G1 + n;
        o.g_d = -1;
        o.u = 0.f;
        o.M_t = s_M[n];
        o.M_d = 0.f;
        o.rho_hi = o.rho_lo = 0.f;
        o.pad = 0;
        o.S_t = (double)s_S[n].hi + (double)s_S[n].lo;
        if (GREEDY) {
            ot[n] = s_arg[n];
        } else if (n < ell) {
            o.mode = 1;
            o.g_d = T1 + b * a.gamma + n;
            o.M_d = s_M[ell + 1 + n];
            const double rho = o.S_t / ((double)s_S[ell + 1 + n].hi + (double)s_S[ell + 1 + n].lo);
            o.rho_hi = (float)rho;
            o.rho_lo = (float)(rho - (double)o.rho_hi);
            o.u = a.uniforms[(size_t)b * (a.gamma + 2) + a.gamma];
        } else {
            o.mode = 2;
            o.u = a.uniforms[(size_t)b * (a.gamma + 2) + a.gamma + 1];
        }
        req[b] = o;
    }
}

// ===================================================================== draw
struct DrawArgs {
    const char* target;
    const char* draft;
    int32_t* out_tokens;
    int B, gamma, V;
    float c_hi, c_lo;
    char* ws;
};

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

// Sum of the weights of one 16-byte vector pair.
template <int ES>
__device__ __forceinline__ float vec_weight_sum(const ReqState& rs, const uint4& t, const uint4& d, float c_hi,
                                                float c_lo) {
    const uint32_t tw[4] = {t.x, t.y, t.z, t.w}, dw[4] = {d.x, d.y, d.z, d.w};
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        if (ES == 2) {
            s0 += draw_weight(rs, bf16_lo(tw[k]), bf16_lo(dw[k]), c_hi, c_lo);
            s1 += draw_weight(rs, bf16_hi(tw[k]), bf16_hi(dw[k]), c_hi, c_lo);
        } else {
            s0 += draw_weight(rs, __uint_as_float(tw[k]), __uint_as_float(dw[k]), c_hi, c_lo);
        }
    }
    return s0 + s1;
}

// Sum of the draw weights over elements [e0, e1) of the draw rows (one warp).
template <int ES>
__device__ float chunk_weight_sum(const ReqState& rs, const char* rt, const char* rd, int e0, int e1, int lane,
                                  float c_hi, float c_lo) {
    constexpr int EPV = 16 / ES;
    constexpr int HALF = kVecPerLane / 2;
    const ChunkSpan st = chunk_span<ES>(rt, e0, e1);
    bool vec = st.ia < st.ib;
    if (rs.mode == 1 && vec) {
        const ChunkSpan sd = chunk_span<ES>(rd, e0, e1);
        vec = sd.ia == st.ia && sd.ib == st.ib;  // same alignment in both rows
    }
    float acc = 0.f;
    if (vec) {
        const int nvec = (st.ib - st.ia) / EPV;  // <= 32 * kVecPerLane
        const uint4* vt = (const uint4*)(rt + (size_t)st.ia * ES);
        const uint4* vd = (const uint4*)(rd + (size_t)st.ia * ES);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint4 tv[HALF], dv[HALF];
#pragma unroll
            for (int k = 0; k < HALF; ++k) {
                const int i = lane + 32 * (h * HALF + k);
                tv[k] = make_uint4(0, 0, 0, 0);
                dv[k] = make_uint4(0, 0, 0, 0);
                if (i < nvec) {
                    tv[k] = __ldg(vt + i);
                    if (rs.mode == 1) dv[k] = __ldg(vd + i);
                }
            }
#pragma unroll
            for (int k = 0; k < HALF; ++k)
                if (lane + 32 * (h * HALF + k) < nvec) acc += vec_weight_sum<ES>(rs, tv[k], dv[k], c_hi, c_lo);
        }
        const int si = span_scalar_index(st, lane);
        if (si >= 0) acc += draw_weight_at<ES>(rs, rt, rd, si, c_hi, c_lo);
    } else {
        for (int i = e0 + lane; i < e1; i += 32) acc += draw_weight_at<ES>(rs, rt, rd, i, c_hi, c_lo);
    }
    return warp_sum(acc);
}

// Inverse-CDF draw inside one chunk: the smallest element index whose running
// weight (from 0 at the chunk start) exceeds r; if none, the last element with
// positive weight (*no_bin set).  One warp.  Lane l owns a contiguous segment;
// lane sums are fp32 (at most 64 terms), the prefix over lanes fp64; the
// crossing segment is then re-read (L2) with its elements spread over the warp
// for a second scan.
template <int ES>
__device__ int chunk_pick(const ReqState& rs, const char* rt, const char* rd, int e0, int e1, double r, int lane,
                          float c_hi, float c_lo, bool* no_bin) {
    constexpr int EPV = 16 / ES;
    constexpr int SEG = kVecPerLane * EPV;  // elements per lane segment (64 bf16 / 32 fp32)
    constexpr int EPL = SEG / 32;           // of those, per lane in the second scan
    constexpr int HALF = kVecPerLane / 2;
    const uint4* vt = (const uint4*)(rt + (size_t)e0 * ES);
    const uint4* vd = (const uint4*)(rd + (size_t)e0 * ES);
    // vector path: a full, 16-byte-aligned chunk; lane l owns vectors [8l, 8l+8)
    const bool full = (e1 - e0) * ES == kChunkBytes && (((uintptr_t)vt & 15) == 0) &&
                      (rs.mode != 1 || (((uintptr_t)vd & 15) == 0));
    float lsum = 0.f;
    int lpos = -1;
    int s0, s1;
    if (full) {
        s0 = e0 + lane * SEG;
        s1 = s0 + SEG;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint4 tv[HALF], dv[HALF];
#pragma unroll
            for (int k = 0; k < HALF; ++k) {
                tv[k] = __ldcg(vt + lane * kVecPerLane + h * HALF + k);
                dv[k] = rs.mode == 1 ? __ldcg(vd + lane * kVecPerLane + h * HALF + k) : make_uint4(0, 0, 0, 0);
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
        const int seg = (e1 - e0 + 31) / 32;
        s0 = min(e1, e0 + lane * seg);
        s1 = min(e1, s0 + seg);
        for (int i = s0; i < s1; ++i) {
            const float w = draw_weight_at<ES>(rs, rt, rd, i, c_hi, c_lo);
            lsum += w;
            if (w > 0.f) lpos = i;
        }
    }
    double excl = (double)lsum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double t = __shfl_up_sync(0xffffffffu, excl, o);
        if (lane >= o) excl += t;
    }
    excl -= (double)lsum;
    const unsigned cross = __ballot_sync(0xffffffffu, s0 < s1 && excl + (double)lsum > r);
    if (!cross) {
        int lp = lpos;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lp = max(lp, __shfl_xor_sync(0xffffffffu, lp, o));
        *no_bin = true;
        return lp >= 0 ? lp : e1 - 1;
    }
    *no_bin = false;
    const int l = __ffs(cross) - 1;
    const float rr = (float)(r - __shfl_sync(0xffffffffu, excl, l));  // remainder inside segment l
    const int seg0 = __shfl_sync(0xffffffffu, s0, l);
    const int seg1 = __shfl_sync(0xffffffffu, s1, l);
    const int segpos = __shfl_sync(0xffffffffu, lpos, l);
    if (full) {
        // lane i takes elements [i*EPL, (i+1)*EPL) of segment l
        float w[EPL];
        float part = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            const int i = seg0 + lane * EPL + e;
            w[e] = draw_weight_at<ES>(rs, rt, rd, i, c_hi, c_lo);
            part += w[e];
        }
        float incl = part;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        const unsigned hit = __ballot_sync(0xffffffffu, incl > rr);
        if (hit) {
            const int i = __ffs(hit) - 1;
            int v = -1;
            if (lane == i) {
                float cum = incl - part;
#pragma unroll
                for (int e = 0; e < EPL; ++e) {
                    cum += w[e];
                    if (v < 0 && cum > rr) v = e;
                }
                if (v < 0) v = EPL - 1;
                v += seg0 + lane * EPL;
            }
            return __shfl_sync(0xffffffffu, v, i);
        }
        return segpos >= 0 ? segpos : seg1 - 1;
    }
    int v = -1;
    if (lane == l) {
        float cum = 0.f;
        for (int i = s0; i < s1 && v < 0; ++i) {
            cum += draw_weight_at<ES>(rs, rt, rd, i, c_hi, c_lo);
            if (cum > rr) v = i;
        }
        if (v < 0) v = lpos >= 0 ? lpos : s1 - 1;
    }
    return __shfl_sync(0xffffffffu, v, l);
}

// Weight total of chunk c of the draw: the residual sums written by the draw
// warps, or, for a bonus draw, the streaming kernel's chunk sums rescaled
// exactly to the row scale.
__device__ __forceinline__ float chunk_total(const ReqState& rs, const float* rchunk, const float2* tpart, int c) {
    if (rs.mode == 1) return __ldcg(rchunk + c);
    const float2 p = tpart[c];
    if (p.x == -INFINITY) return 0.f;
    const float d = p.x - rs.M_t;
    return p.y * pow2_f(d < -1000.f ? -1000 : (int)d);
}

// One warp per (request, chunk): residual chunk sums.  The warp that completes
// a request's last chunk (per-request ticket, zeroed by the accept kernel of
// the same call) then draws the token: fp64 prefix over the chunk totals, then
// chunk_pick inside the chosen chunk.  A bonus draw needs no pass over the row:
// the warp of chunk 0 draws directly from the streaming kernel's chunk sums.
constexpr int kDrawWarps = 8;

template <int ES>
__global__ void __launch_bounds__(kDrawWarps * 32, 4) k_draw(DrawArgs a, Layout L) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long item = (long long)blockIdx.x * kDrawWarps + warp;
    pdl_wait();
    if (item >= (long long)a.B * L.nch) return;
    const int b = (int)(item / L.nch), c = (int)(item - (long long)b * L.nch);
    ReqState rs = ((const ReqState*)(a.ws + L.req))[b];
    if (rs.status != SPEC_OK || rs.mode == 0) return;
    if (rs.mode == 2 && c != 0) return;
    int* hdr = (int*)(a.ws + L.hdr);
    const int T1 = a.B * (a.gamma + 1);
    const char* rt = a.target + (size_t)rs.g_t * a.V * ES;
    const char* rd = rs.mode == 1 ? a.draft + (size_t)(rs.g_d - T1) * a.V * ES : rt;
    float* rchunk = (float*)(a.ws + L.rchunk) + (size_t)b * L.nch;
    const float2* tpart = (const float2*)(a.ws + L.partial) + (size_t)rs.g_t * L.nch;

    if (rs.mode == 1) {
        const int e0 = c * L.CH, e1 = min(a.V, e0 + L.CH);
        const float sum = chunk_weight_sum<ES>(rs, rt, rd, e0, e1, lane, a.c_hi, a.c_lo);
        int last = 0;
        if (lane == 0) {
            rchunk[c] = sum;
            __threadfence();
            last = atomicAdd((int*)(a.ws + L.ticket) + b, 1) == L.nch - 1;
        }
        if (!__shfl_sync(0xffffffffu, last, 0)) return;
        __threadfence();
    }

    // this warp draws the request's token
    double W = 0.0;
    for (int k = lane; k < L.nch; k += 32) W += (double)chunk_total(rs, rchunk, tpart, k);
    W = warp_sum_d(W);
    if (!(W > 0.0) && rs.mode == 1) {
        // the residual summed to zero: draw from p of the same row instead
        rs.mode = 2;
        rd = rt;
        if (lane == 0) atomicOr(&hdr[kHdrEvents], 1);
        W = 0.0;
        for (int k = lane; k < L.nch; k += 32) W += (double)chunk_total(rs, rchunk, tpart, k);
        W = warp_sum_d(W);
    }
    const double target = (double)rs.u * W;
    // first chunk whose inclusive fp64 prefix exceeds u * W
    int cstar = -1, last_pos = -1;
    double before = 0.0, run = 0.0;
    for (int base = 0; base < L.nch && cstar < 0; base += 32) {
        const int k = base + lane;
        const double v = k < L.nch ? (double)chunk_total(rs, rchunk, tpart, k) : 0.0;
        double incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        incl += run;
        const unsigned hit = __ballot_sync(0xffffffffu, k < L.nch && incl > target);
        const unsigned pos = __ballot_sync(0xffffffffu, k < L.nch && v > 0.0);
        if (pos) last_pos = base + 31 - __clz(pos);
        if (hit) {
            const int l = __ffs(hit) - 1;
            cstar = base + l;
            before = __shfl_sync(0xffffffffu, incl - v, l);
        }
        run = __shfl_sync(0xffffffffu, incl, 31);
    }
    bool force_last = false;
    if (cstar < 0) {  // rounding left no chunk: the last chunk with positive weight
        cstar = last_pos >= 0 ? last_pos : L.nch - 1;
        force_last = true;
    }
    const double r = force_last ? INFINITY : target - before;
    const int e0 = cstar * L.CH, e1 = min(a.V, e0 + L.CH);
    bool no_bin = false;
    const int tok = chunk_pick<ES>(rs, rt, rd, e0, e1, r, lane, a.c_hi, a.c_lo, &no_bin);
    if (lane == 0) {
        a.out_tokens[(size_t)b * (a.gamma + 1) + rs.n] = tok;
        ((double*)(a.ws + L.mass))[b] = W / rs.S_t;
        if (no_bin && !force_last) atomicOr(&hdr[kHdrEvents], 2);
    }
}

// ==================================================================== stats
__global__ void k_copy_stats(const char* ws, Layout L, int B, int gamma, double* px, double* qx,
                             double* mass, int32_t* status) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    const double* pq = (const double*)(ws + L.pq);
    if (i < B * gamma) {
        if (px) px[i] = pq[2 * (size_t)i];
        if (qx) qx[i] = pq[2 * (size_t)i + 1];
    }
    if (i < B) {
        const ReqState rs = ((const ReqState*)(ws + L.req))[i];
        if (mass) mass[i] = rs.status == SPEC_OK ? ((const double*)(ws + L.mass))[i]
                                                 : __longlong_as_double(0x7ff8000000000000ll);
        if (status) status[i] = rs.status;
    }
}

}  // namespace specv

// ===================================================================== host
using namespace specv;

namespace {

cudaEvent_t g_ev_before = nullptr, g_ev_after = nullptr;

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
        const void* fns[8] = {
            (const void*)k_row_stats<2, false, false>, (const void*)k_row_stats<2, true, false>,
            (const void*)k_row_stats<4, false, false>, (const void*)k_row_stats<4, true, false>,
            (const void*)k_row_stats<2, false, true>,  (const void*)k_row_stats<2, true, true>,
            (const void*)k_row_stats<4, false, true>,  (const void*)k_row_stats<4, true, true>};
        for (const void* f : fns)
            if (cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kStatsSmem) !=
                cudaSuccess)
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
int launch_chain(const StatsArgs& sa, const AcceptArgs& aa, const DrawArgs& da, const Layout& L, int sms,
                 bool aligned_rows, cudaStream_t st) {
    const long long max_items = (long long)L.R * L.nch;
    const int grid = (int)std::min<long long>(sms, (max_items + kStatsWarps - 1) / kStatsWarps);
    if (g_ev_before) cudaEventRecord(g_ev_before, st);
    if (aligned_rows)
        k_row_stats<ES, GREEDY, true><<<grid, kStatsThreads, kStatsSmem, st>>>(sa, L);
    else
        k_row_stats<ES, GREEDY, false><<<grid, kStatsThreads, kStatsSmem, st>>>(sa, L);
    if (g_ev_after) cudaEventRecord(g_ev_after, st);
    // the accept and draw kernels may be scheduled while their predecessor
    // finishes; they wait for its results with griddepcontrol.wait
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)sa.B);
    cfg.blockDim = dim3(kReqThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, k_accept<ES, GREEDY>, aa, L) != cudaSuccess) return SPEC_ERR_CUDA;
    if (!GREEDY) {
        const long long items = (long long)sa.B * L.nch;
        cfg.gridDim = dim3((unsigned)((items + kDrawWarps - 1) / kDrawWarps));
        cfg.blockDim = dim3(kDrawWarps * 32);
        if (cudaLaunchKernelEx(&cfg, k_draw<ES>, da, L) != cudaSuccess) return SPEC_ERR_CUDA;
    }
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
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
    StatsArgs sa{t, d, verify_len, B, gamma, V, c_hi, c_lo, ws};
    AcceptArgs aa{t, d, draft_tokens, verify_len, uniforms, out_tokens, out_accept_len, B, gamma, V, c_hi, c_lo, ws};
    DrawArgs da{t, d, out_tokens, B, gamma, V, c_hi, c_lo, ws};
    cudaStream_t st = (cudaStream_t)stream;
    // every row starts on a 16-byte boundary: whole-chunk copies
    const bool al = aligned(target_logits, 16) && (greedy || gamma == 0 || aligned(draft_logits, 16)) &&
                    ((size_t)V * es) % 16 == 0;
    if (es == 2)
        return greedy ? launch_chain<2, true>(sa, aa, da, L, sms, al, st)
                      : launch_chain<2, false>(sa, aa, da, L, sms, al, st);
    return greedy ? launch_chain<4, true>(sa, aa, da, L, sms, al, st)
                  : launch_chain<4, false>(sa, aa, da, L, sms, al, st);
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
    g_ev_before = (cudaEvent_t)before_row_stats;
    g_ev_after = (cudaEvent_t)after_row_stats;
    return SPEC_OK;
}

int spec_verify_kernel_count(int B, float temperature) {
    if (B <= 0) return 0;
    return temperature == 0.0f ? 2 : 3;
}

}  // extern "C"
