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
//   k_plan       1 CTA: validates requests, lists the needed logit rows.
//   k_row_stats  persistent, one CTA per SM: the HBM pass.  Each warp streams
//                4 KiB row chunks through its own ring of shared-memory stages
//                filled by 1-D bulk copies (cp.async.bulk + mbarrier) and
//                writes per-chunk (scale, sum) or (max, argmax) partials.
//   k_accept     1 CTA per request: merges chunk partials per row (exact
//                power-of-two rescaling, fp64 sums), computes p(x), q(x), runs
//                the accept tests with a warp ballot, writes the accepted
//                prefix and the draw job.
//   k_resid_sum  one warp per (request, chunk): residual / bonus chunk sums
//                over the 1-2 draw rows of each request.
//   k_resid_pick one warp per request: fp64 prefix over chunk sums, then an
//                in-chunk scan for the inverse-CDF draw.
#include <math.h>

#include <algorithm>
#include <mutex>

#include "specv_common.cuh"

namespace specv {

// ===================================================================== plan
// Per request: validate verify_len, the draft tokens and (T > 0) the used
// uniforms; count needed rows (target 0..ell, draft 0..ell-1) and list them.
__global__ void __launch_bounds__(1024) k_plan(const int32_t* __restrict__ verify_len,
                                               const int32_t* __restrict__ tokens,
                                               const float* __restrict__ uniforms, int B,
                                               int gamma, int V, int greedy,
                                               int32_t* __restrict__ out_tokens,
                                               int32_t* __restrict__ out_accept_len, char* ws,
                                               Layout L) {
    __shared__ int s_warp[32];
    __shared__ int s_total;
    int* hdr = (int*)(ws + L.hdr);
    ReqState* req = (ReqState*)(ws + L.req);
    int* row_list = (int*)(ws + L.row_list);
    double* pq = (double*)(ws + L.pq);
    double* mass = (double*)(ws + L.mass);

    const int tid = threadIdx.x;
    if (tid == 0) {
        hdr[kHdrStatus] = 0;
        hdr[kHdrEvents] = 0;
    }
    __syncthreads();

    constexpr int PER = 4;  // requests per thread (B <= 4096)
    int cnt[PER];
    int ells[PER];
    int mine = 0;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int b = tid * PER + i;
        cnt[i] = 0;
        ells[i] = 0;
        if (b >= B) continue;
        int st = SPEC_OK;
        const int ell = verify_len ? verify_len[b] : gamma;
        if (ell < 0 || ell > gamma) st = SPEC_ERR_VERIFY_LEN;
        if (st == SPEC_OK)
            for (int j = 0; j < ell; ++j) {
                const int x = tokens[(size_t)b * gamma + j];
                if (x < 0 || x >= V) { st = SPEC_ERR_TOKEN; break; }
            }
        if (st == SPEC_OK && !greedy) {
            const float* u = uniforms + (size_t)b * (gamma + 2);
            for (int j = 0; j < ell; ++j)
                if (!(u[j] >= 0.0f && u[j] < 1.0f)) st = SPEC_ERR_UNIFORM;
            if (!(u[gamma] >= 0.0f && u[gamma] < 1.0f) || !(u[gamma + 1] >= 0.0f && u[gamma + 1] < 1.0f))
                st = SPEC_ERR_UNIFORM;
        }
        ReqState rs;
        rs.ell = st == SPEC_OK ? ell : 0;
        rs.status = st;
        rs.n = -1;
        rs.mode = 0;
        rs.g_t = rs.g_d = -1;
        rs.u = 0.f;
        rs.M_t = rs.M_d = 0.f;
        rs.rho_hi = rs.rho_lo = 0.f;
        rs.pad = 0;
        rs.S_t = 0.0;
        req[b] = rs;
        for (int j = 0; j < gamma; ++j) {
            pq[2 * ((size_t)b * gamma + j)] = __longlong_as_double(0x7ff8000000000000ll);
            pq[2 * ((size_t)b * gamma + j) + 1] = __longlong_as_double(0x7ff8000000000000ll);
        }
        mass[b] = __longlong_as_double(0x7ff8000000000000ll);
        if (st != SPEC_OK) {
            for (int j = 0; j <= gamma; ++j) out_tokens[(size_t)b * (gamma + 1) + j] = -1;
            out_accept_len[b] = -1;
            set_status(&hdr[kHdrStatus], st);
        } else {
            ells[i] = ell;
            cnt[i] = greedy ? ell + 1 : 2 * ell + 1;
        }
        mine += cnt[i];
    }

    // block-wide exclusive scan of `mine`
    const int lane = tid & 31, warp = tid >> 5;
    int incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = lane < (int)(blockDim.x >> 5) ? s_warp[lane] : 0;
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += v;
        }
        s_warp[lane] = wi - w;
        if (lane == 31) s_total = wi;
    }
    __syncthreads();
    int off = s_warp[warp] + incl - mine;
    const int T1 = B * (gamma + 1);
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int b = tid * PER + i;
        if (b >= B || cnt[i] == 0) continue;
        for (int j = 0; j <= ells[i]; ++j) row_list[off++] = b * (gamma + 1) + j;
        if (!greedy)
            for (int j = 0; j < ells[i]; ++j) row_list[off++] = T1 + b * gamma + j;
    }
    if (tid == 0) hdr[kHdrRows] = s_total;
}

// ================================================================ row stats
// One work item = one chunk (kChunkBytes) of one needed row, handled by one
// warp.  The aligned interior arrives through a bulk copy into the warp's ring
// stage; up to 15 head and 7 tail elements are loaded directly by lanes.
template <int ES, bool GREEDY>
__device__ __forceinline__ float2 chunk_stats(const char* stage, const ChunkSpan& sp, int lane,
                                              float c_hi, float c_lo) {
    constexpr int EPV = 16 / ES;  // elements per 16-byte vector
    const int nvec = (sp.ib - sp.ia) / EPV;
    const uint4* sm = (const uint4*)stage;
    const int si = span_scalar_index(sp, lane);
    const float sv = si >= 0 ? load_logit<ES>(sp.rowp, si) : -INFINITY;

    // pass 1: max (NaN-propagating)
    float m;
    if (ES == 2) {
        uint32_t pm = 0xFF80FF80u;  // (-inf, -inf)
        int i = lane;
        for (; i + 32 < nvec; i += 64) {
            const uint4 a = sm[i], b = sm[i + 32];
            pm = bf16x2_max_nan(pm, bf16x2_max_nan(bf16x2_max_nan(a.x, a.y), bf16x2_max_nan(a.z, a.w)));
            pm = bf16x2_max_nan(pm, bf16x2_max_nan(bf16x2_max_nan(b.x, b.y), bf16x2_max_nan(b.z, b.w)));
        }
        if (i < nvec) {
            const uint4 a = sm[i];
            pm = bf16x2_max_nan(pm, bf16x2_max_nan(bf16x2_max_nan(a.x, a.y), bf16x2_max_nan(a.z, a.w)));
        }
        m = fmax_nan(bf16_lo(pm), bf16_hi(pm));
    } else {
        m = -INFINITY;
        for (int i = lane; i < nvec; i += 32) {
            const float4 a = ((const float4*)stage)[i];
            m = fmax_nan(m, fmax_nan(fmax_nan(a.x, a.y), fmax_nan(a.z, a.w)));
        }
    }
    m = fmax_nan(m, sv);
    m = warp_max_nan(m);

    if (GREEDY) {
        // lowest index attaining the max
        int best = 0x7fffffff;
        if (!(m != m)) {
            for (int i = lane; i < nvec && best == 0x7fffffff; i += 32) {
                const int base = sp.ia + i * EPV;
                if (ES == 2) {
                    const uint4 a = sm[i];
                    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        if (best == 0x7fffffff && bf16_lo(w[k]) == m) best = base + 2 * k;
                        if (best == 0x7fffffff && bf16_hi(w[k]) == m) best = base + 2 * k + 1;
                    }
                } else {
                    const float4 a = ((const float4*)stage)[i];
                    const float w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        if (best == 0x7fffffff && w[k] == m) best = base + k;
                }
            }
            if (si >= 0 && sv == m) best = min(best, si);
        }
        best = warp_min_i(best);
        return make_float2(m, __int_as_float(best));
    }

    // T > 0
    if (m != m || m == INFINITY) return make_float2(__int_as_float(0x7fc00000), 0.f);
    if (m == -INFINITY) return make_float2(-INFINITY, 0.f);
    const float Mc = ceilf(fmaf(m, c_hi, m * c_lo));
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
    if (ES == 2) {
        for (int i = lane; i < nvec; i += 32) {
            const uint4 a = sm[i];
            a0 += scaled_exp(bf16_lo(a.x), c_hi, c_lo, Mc);
            a1 += scaled_exp(bf16_hi(a.x), c_hi, c_lo, Mc);
            a2 += scaled_exp(bf16_lo(a.y), c_hi, c_lo, Mc);
            a3 += scaled_exp(bf16_hi(a.y), c_hi, c_lo, Mc);
            a0 += scaled_exp(bf16_lo(a.z), c_hi, c_lo, Mc);
            a1 += scaled_exp(bf16_hi(a.z), c_hi, c_lo, Mc);
            a2 += scaled_exp(bf16_lo(a.w), c_hi, c_lo, Mc);
            a3 += scaled_exp(bf16_hi(a.w), c_hi, c_lo, Mc);
        }
    } else {
        for (int i = lane; i < nvec; i += 32) {
            const float4 a = ((const float4*)stage)[i];
            a0 += scaled_exp(a.x, c_hi, c_lo, Mc);
            a1 += scaled_exp(a.y, c_hi, c_lo, Mc);
            a2 += scaled_exp(a.z, c_hi, c_lo, Mc);
            a3 += scaled_exp(a.w, c_hi, c_lo, Mc);
        }
    }
    if (si >= 0) a0 += scaled_exp(sv, c_hi, c_lo, Mc);
    const float S = warp_sum((a0 + a1) + (a2 + a3));
    return make_float2(Mc, S);
}

struct StatsArgs {
    const char* target;
    const char* draft;
    int B, gamma, V;
    float c_hi, c_lo;
    char* ws;
};

template <int ES, bool GREEDY>
__global__ void __launch_bounds__(kStatsWarps * 32, 1) k_row_stats(StatsArgs a, Layout L) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = (unsigned char*)(((uintptr_t)smem_raw + 127) & ~uintptr_t(127));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    unsigned char* ring = smem + (size_t)warp * kStages * kChunkBytes;
    uint64_t* bars = (uint64_t*)(smem + (size_t)kStatsWarps * kStages * kChunkBytes) + warp * kStages;

    int* hdr = (int*)(a.ws + L.hdr);
    const int* row_list = (const int*)(a.ws + L.row_list);
    float2* partial = (float2*)(a.ws + L.partial);

    if (lane == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncwarp();

    const long long total = (long long)hdr[kHdrRows] * L.nch;
    const long long W = (long long)gridDim.x * kStatsWarps;
    const long long first = (long long)blockIdx.x * kStatsWarps + warp;
    const int T1 = a.B * (a.gamma + 1);

    auto span_of = [&](long long item, int& g, int& c) -> ChunkSpan {
        const int r = (int)(item / L.nch);
        c = (int)(item - (long long)r * L.nch);
        g = row_list[r];
        const char* rowp = g < T1 ? a.target + (size_t)g * a.V * ES
                                  : a.draft + (size_t)(g - T1) * a.V * ES;
        const int e0 = c * L.CH;
        const int e1 = min(a.V, e0 + L.CH);
        return chunk_span<ES>(rowp, e0, e1);
    };
    auto issue = [&](int s, long long item) {
        int g, c;
        const ChunkSpan sp = span_of(item, g, c);
        if (sp.ia < sp.ib && lane == 0) {
            const uint32_t bytes = (uint32_t)((sp.ib - sp.ia) * ES);
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&bars[s], bytes);
            bulk_g2s(ring + (size_t)s * kChunkBytes, sp.rowp + (size_t)sp.ia * ES, bytes, &bars[s]);
        }
        return sp.ia < sp.ib;
    };

    uint32_t phase = 0;     // bit s: parity of the next wait on stage s
    uint32_t pending = 0;   // bit s: a copy is in flight on stage s
#pragma unroll 1
    for (int s = 0; s < kStages; ++s) {
        const long long item = first + (long long)s * W;
        if (item < total && issue(s, item)) pending |= 1u << s;
    }

    int s = 0;
    bool timed_out = false;
#pragma unroll 1
    for (long long item = first; item < total; item += W) {
        int g, c;
        const ChunkSpan sp = span_of(item, g, c);
        const unsigned char* stage = ring + (size_t)s * kChunkBytes;
        if (pending & (1u << s)) {
            if (!mbar_wait_bounded(&bars[s], (phase >> s) & 1u)) {
                timed_out = true;
                break;
            }
            phase ^= 1u << s;
            pending &= ~(1u << s);
        }
        const float2 r = chunk_stats<ES, GREEDY>((const char*)stage, sp, lane, a.c_hi, a.c_lo);
        if (lane == 0) partial[(size_t)g * L.nch + c] = r;
        __syncwarp();
        const long long next = item + (long long)kStages * W;
        if (next < total && issue(s, next)) pending |= 1u << s;
        s = (s + 1 == kStages) ? 0 : s + 1;
    }

    if (timed_out) {
        // Record the failure, let copies in flight land (bounded), and mark
        // every item this warp did not finish as invalid.
        if (lane == 0) set_status(&hdr[kHdrStatus], SPEC_ERR_TIMEOUT);
        for (int k = 0; k < kStages; ++k)
            if (pending & (1u << k)) mbar_wait_bounded(&bars[k], (phase >> k) & 1u);
        for (long long item = first; item < total; item += W) {
            const int r = (int)(item / L.nch);
            const int c = (int)(item - (long long)r * L.nch);
            if (lane == 0)
                partial[(size_t)row_list[r] * L.nch + c] = make_float2(__int_as_float(0x7fc00000), 0.f);
        }
    }
}

// =================================================================== accept
struct AcceptArgs {
    const char* target;
    const char* draft;
    const int32_t* tokens;
    const float* uniforms;
    int32_t* out_tokens;
    int32_t* out_accept_len;
    int B, gamma, V;
    float c_hi, c_lo;
    char* ws;
};

// Merge the chunk partials of row g into a RowStat.
template <bool GREEDY>
__device__ __forceinline__ RowStat merge_row(const float2* part, int nch, int lane) {
    RowStat rs;
    rs.arg = 0;
    if (GREEDY) {
        float best = -INFINITY;
        int arg = 0x7fffffff;
        bool bad = false;
        for (int c = lane; c < nch; c += 32) {
            const float2 p = part[c];
            const int ix = __float_as_int(p.y);
            if (p.x != p.x) bad = true;
            else if (p.x > best || (p.x == best && ix < arg)) { best = p.x; arg = ix; }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ob = __shfl_xor_sync(0xffffffffu, best, o);
            const int oa = __shfl_xor_sync(0xffffffffu, arg, o);
            if (ob > best || (ob == best && oa < arg)) { best = ob; arg = oa; }
        }
        bad = __any_sync(0xffffffffu, bad);
        rs.M = best;
        rs.arg = arg;
        rs.S = (bad || !(fabsf(best) <= 3.402823466e38f)) ? __longlong_as_double(0x7ff8000000000000ll) : 1.0;
        return rs;
    }
    float M = -INFINITY;
    for (int c = lane; c < nch; c += 32) M = fmax_nan(M, part[c].x);
    M = warp_max_nan(M);
    rs.M = M;
    if (M != M || M == -INFINITY) {
        rs.S = __longlong_as_double(0x7ff8000000000000ll);
        return rs;
    }
    double S = 0.0;
    for (int c = lane; c < nch; c += 32) {
        const float2 p = part[c];
        if (p.x != -INFINITY) {
            // M and p.x are integer-valued floats: the rescale is an exact power of two
            const float d = p.x - M;
            const int e = d < -1000.f ? -1000 : (int)d;
            S += ldexp((double)p.y, e);
        }
    }
    rs.S = warp_sum_d(S);
    return rs;
}

template <int ES, bool GREEDY>
__global__ void __launch_bounds__(128) k_accept(AcceptArgs a, Layout L) {
    const int b = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int* hdr = (int*)(a.ws + L.hdr);
    ReqState* req = (ReqState*)(a.ws + L.req);
    const float2* partial = (const float2*)(a.ws + L.partial);
    RowStat* rstat = (RowStat*)(a.ws + L.row_stat);
    double* pq = (double*)(a.ws + L.pq);
    __shared__ int s_bad;

    ReqState rs = req[b];
    if (rs.status != SPEC_OK) return;
    const int ell = rs.ell, G1 = a.gamma + 1, T1 = a.B * G1;
    if (threadIdx.x == 0) s_bad = 0;
    __syncthreads();

    const int nrows = GREEDY ? ell + 1 : 2 * ell + 1;
    for (int r = warp; r < nrows; r += 4) {
        const int g = r <= ell ? b * G1 + r : T1 + b * a.gamma + (r - ell - 1);
        const RowStat st = merge_row<GREEDY>(partial + (size_t)g * L.nch, L.nch, lane);
        if (lane == 0) {
            rstat[g] = st;
            if (st.S != st.S) s_bad = 1;
        }
    }
    __syncthreads();
    if (warp != 0) return;

    const int32_t* x = a.tokens + (size_t)b * a.gamma;
    int32_t* ot = a.out_tokens + (size_t)b * G1;
    if (s_bad) {
        for (int j = lane; j <= a.gamma; j += 32) ot[j] = -1;
        if (lane == 0) {
            a.out_accept_len[b] = -1;
            req[b].status = SPEC_ERR_NONFINITE;
            set_status(&hdr[kHdrStatus], SPEC_ERR_NONFINITE);
        }
        return;
    }

    // accept tests, one lane per position (gamma <= 32)
    bool acc = true;
    const int j = lane;
    if (j < ell) {
        const int xj = x[j];
        const int gt = b * G1 + j;
        if (GREEDY) {
            acc = xj == rstat[gt].arg;
        } else {
            const int gd = T1 + b * a.gamma + j;
            const RowStat st = rstat[gt], sd = rstat[gd];
            const float zt = load_logit<ES>(a.target + (size_t)gt * a.V * ES, xj);
            const float zd = load_logit<ES>(a.draft + (size_t)(gd - T1) * a.V * ES, xj);
            const double px = (double)scaled_exp(zt, a.c_hi, a.c_lo, st.M) / st.S;
            const double qx = (double)scaled_exp(zd, a.c_hi, a.c_lo, sd.M) / sd.S;
            pq[2 * ((size_t)b * a.gamma + j)] = px;
            pq[2 * ((size_t)b * a.gamma + j) + 1] = qx;
            const double u = (double)a.uniforms[(size_t)b * (a.gamma + 2) + j];
            acc = u * qx < px;
        }
    }
    const unsigned rej = __ballot_sync(0xffffffffu, !acc);
    const int n = rej ? min(__ffs(rej) - 1, ell) : ell;
    for (int k = lane; k <= a.gamma; k += 32) {
        if (k < n) ot[k] = x[k];
        else if (k > n) ot[k] = -1;
    }
    if (lane == 0) {
        a.out_accept_len[b] = n;
        req[b].n = n;
        if (GREEDY) {
            ot[n] = rstat[b * G1 + n].arg;
        } else {
            const int gt = b * G1 + n;
            const RowStat st = rstat[gt];
            ReqState o = rs;
            o.n = n;
            o.g_t = gt;
            o.M_t = st.M;
            o.S_t = st.S;
            if (n < ell) {
                const int gd = T1 + b * a.gamma + n;
                const RowStat sd = rstat[gd];
                o.mode = 1;
                o.g_d = gd;
                o.M_d = sd.M;
                const double rho = st.S / sd.S;
                o.rho_hi = (float)rho;
                o.rho_lo = (float)(rho - (double)o.rho_hi);
                o.u = a.uniforms[(size_t)b * (a.gamma + 2) + a.gamma];
            } else {
                o.mode = 2;
                o.g_d = -1;
                o.u = a.uniforms[(size_t)b * (a.gamma + 2) + a.gamma + 1];
            }
            req[b] = o;
        }
    }
}

// ================================================================= residual
struct ResidArgs {
    const char* target;
    const char* draft;
    int32_t* out_tokens;
    int B, gamma, V;
    float c_hi, c_lo;
    char* ws;
};

// Weight of element i of the draw: residual max(e_t - rho * e_d, 0) (both
// relative to their rows' scales) or the target weight e_t.
template <int ES>
__device__ __forceinline__ float draw_weight(const ReqState& rs, const char* rt, const char* rd, int i,
                                             float c_hi, float c_lo) {
    const float et = scaled_exp(load_logit<ES>(rt, i), c_hi, c_lo, rs.M_t);
    if (rs.mode != 1) return et;
    const float ed = scaled_exp(load_logit<ES>(rd, i), c_hi, c_lo, rs.M_d);
    return fmaxf(fmaf(-rs.rho_lo, ed, fmaf(-rs.rho_hi, ed, et)), 0.f);
}

template <int ES>
__device__ __forceinline__ float weight_from_pair(const ReqState& rs, float zt, float zd, float c_hi,
                                                  float c_lo) {
    const float et = scaled_exp(zt, c_hi, c_lo, rs.M_t);
    if (rs.mode != 1) return et;
    const float ed = scaled_exp(zd, c_hi, c_lo, rs.M_d);
    return fmaxf(fmaf(-rs.rho_lo, ed, fmaf(-rs.rho_hi, ed, et)), 0.f);
}

// Sum of draw weights over chunk c of request b.
template <int ES>
__device__ float chunk_weight_sum(const ReqState& rs, const char* rt, const char* rd, int e0, int e1,
                                  int lane, float c_hi, float c_lo) {
    constexpr int EPV = 16 / ES;
    ChunkSpan st = chunk_span<ES>(rt, e0, e1);
    bool vec = st.ia < st.ib;
    if (rs.mode == 1 && vec) {
        const ChunkSpan sd = chunk_span<ES>(rd, e0, e1);
        vec = sd.ia == st.ia && sd.ib == st.ib;  // same alignment in both rows
    }
    float a0 = 0.f, a1 = 0.f;
    if (vec) {
        const int nvec = (st.ib - st.ia) / EPV;
        const uint4* vt = (const uint4*)(rt + (size_t)st.ia * ES);
        const uint4* vd = (const uint4*)(rd + (size_t)st.ia * ES);
        for (int i = lane; i < nvec; i += 32) {
            const uint4 t = __ldg(vt + i);
            uint4 d = make_uint4(0, 0, 0, 0);
            if (rs.mode == 1) d = __ldg(vd + i);
            if (ES == 2) {
                const uint32_t tw[4] = {t.x, t.y, t.z, t.w}, dw[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    a0 += weight_from_pair<ES>(rs, bf16_lo(tw[k]), bf16_lo(dw[k]), c_hi, c_lo);
                    a1 += weight_from_pair<ES>(rs, bf16_hi(tw[k]), bf16_hi(dw[k]), c_hi, c_lo);
                }
            } else {
                a0 += weight_from_pair<ES>(rs, __uint_as_float(t.x), __uint_as_float(d.x), c_hi, c_lo);
                a1 += weight_from_pair<ES>(rs, __uint_as_float(t.y), __uint_as_float(d.y), c_hi, c_lo);
                a0 += weight_from_pair<ES>(rs, __uint_as_float(t.z), __uint_as_float(d.z), c_hi, c_lo);
                a1 += weight_from_pair<ES>(rs, __uint_as_float(t.w), __uint_as_float(d.w), c_hi, c_lo);
            }
        }
        const int si = span_scalar_index(st, lane);
        if (si >= 0) a0 += draw_weight<ES>(rs, rt, rd, si, c_hi, c_lo);
    } else {
        for (int i = e0 + lane; i < e1; i += 32) a0 += draw_weight<ES>(rs, rt, rd, i, c_hi, c_lo);
    }
    return warp_sum(a0 + a1);
}

template <int ES>
__global__ void __launch_bounds__(256) k_resid_sum(ResidArgs a, Layout L) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long item = (long long)blockIdx.x * 8 + warp;
    if (item >= (long long)a.B * L.nch) return;
    const int b = (int)(item / L.nch), c = (int)(item - (long long)b * L.nch);
    const ReqState rs = ((const ReqState*)(a.ws + L.req))[b];
    if (rs.status != SPEC_OK || rs.mode == 0) return;
    const int T1 = a.B * (a.gamma + 1);
    const char* rt = a.target + (size_t)rs.g_t * a.V * ES;
    const char* rd = rs.mode == 1 ? a.draft + (size_t)(rs.g_d - T1) * a.V * ES : rt;
    const int e0 = c * L.CH, e1 = min(a.V, e0 + L.CH);
    const float s = chunk_weight_sum<ES>(rs, rt, rd, e0, e1, lane, a.c_hi, a.c_lo);
    if (lane == 0) ((float*)(a.ws + L.rchunk))[(size_t)b * L.nch + c] = s;
}

template <int ES>
__global__ void __launch_bounds__(128) k_resid_pick(ResidArgs a, Layout L) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.x * 4 + warp;
    if (b >= a.B) return;
    ReqState* reqs = (ReqState*)(a.ws + L.req);
    ReqState rs = reqs[b];
    if (rs.status != SPEC_OK || rs.mode == 0) return;
    int* hdr = (int*)(a.ws + L.hdr);
    const int T1 = a.B * (a.gamma + 1);
    const char* rt = a.target + (size_t)rs.g_t * a.V * ES;
    const char* rd = rs.mode == 1 ? a.draft + (size_t)(rs.g_d - T1) * a.V * ES : rt;
    float* rchunk = (float*)(a.ws + L.rchunk) + (size_t)b * L.nch;

    // total weight; an empty residual falls back to a draw from p of the same row
    double W = 0.0;
    for (int c = lane; c < L.nch; c += 32) W += (double)rchunk[c];
    W = warp_sum_d(W);
    if (!(W > 0.0) && rs.mode == 1) {
        rs.mode = 2;
        if (lane == 0) atomicOr(&hdr[kHdrEvents], 1);
        for (int c = 0; c < L.nch; ++c) {
            const int e0 = c * L.CH, e1 = min(a.V, e0 + L.CH);
            const float s = chunk_weight_sum<ES>(rs, rt, rt, e0, e1, lane, a.c_hi, a.c_lo);
            if (lane == 0) rchunk[c] = s;
        }
        __syncwarp();
        W = 0.0;
        for (int c = lane; c < L.nch; c += 32) W += (double)rchunk[c];
        W = warp_sum_d(W);
    }
    const double target = (double)rs.u * W;

    // first chunk whose inclusive prefix exceeds u * W (fp64 prefix in chunk order)
    int cstar = -1;
    double before = 0.0, run = 0.0;
    int last_pos = -1;
    for (int base = 0; base < L.nch && cstar < 0; base += 32) {
        const int c = base + lane;
        const double v = c < L.nch ? (double)rchunk[c] : 0.0;
        double incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        incl += run;
        const unsigned hit = __ballot_sync(0xffffffffu, c < L.nch && incl > target);
        const unsigned pos = __ballot_sync(0xffffffffu, c < L.nch && v > 0.0);
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
        before = 0.0;
    }
    const double r = force_last ? INFINITY : target - before;

    // in-chunk scan: lane l owns a contiguous segment of the chunk
    const int e0 = cstar * L.CH, e1 = min(a.V, e0 + L.CH);
    const int seg = (e1 - e0 + 31) / 32;
    const int s0 = min(e1, e0 + lane * seg), s1 = min(e1, s0 + seg);
    double lsum = 0.0;
    int lpos = -1;
    for (int i = s0; i < s1; ++i) {
        const float w = draw_weight<ES>(rs, rt, rd, i, a.c_hi, a.c_lo);
        lsum += (double)w;
        if (w > 0.f) lpos = i;
    }
    double excl = lsum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double t = __shfl_up_sync(0xffffffffu, excl, o);
        if (lane >= o) excl += t;
    }
    excl -= lsum;
    const unsigned cross = __ballot_sync(0xffffffffu, excl + lsum > r && s0 < s1);
    int tok;
    if (cross) {
        const int l = __ffs(cross) - 1;
        int v = -1;
        if (lane == l) {
            double cum = excl;
            for (int i = s0; i < s1; ++i) {
                cum += (double)draw_weight<ES>(rs, rt, rd, i, a.c_hi, a.c_lo);
                if (cum > r) { v = i; break; }
            }
            if (v < 0) v = lpos >= 0 ? lpos : s1 - 1;
        }
        tok = __shfl_sync(0xffffffffu, v, l);
    } else {
        int lp = lpos;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lp = max(lp, __shfl_xor_sync(0xffffffffu, lp, o));
        tok = lp >= 0 ? lp : e1 - 1;
        if (lane == 0 && !force_last) atomicOr(&hdr[kHdrEvents], 2);
    }
    if (lane == 0) {
        a.out_tokens[(size_t)b * (a.gamma + 1) + rs.n] = tok;
        ((double*)(a.ws + L.mass))[b] = W / rs.S_t;
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
        const void* fns[4] = {(const void*)k_row_stats<2, false>, (const void*)k_row_stats<2, true>,
                              (const void*)k_row_stats<4, false>, (const void*)k_row_stats<4, true>};
        for (const void* f : fns)
            if (cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, kStatsSmem) !=
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
int launch_chain(const StatsArgs& sa, const AcceptArgs& aa, const ResidArgs& ra,
                 const int32_t* verify_len, const int32_t* tokens, const float* uniforms,
                 int32_t* out_tokens, int32_t* out_accept_len, const Layout& L, int sms,
                 cudaStream_t st) {
    k_plan<<<1, 1024, 0, st>>>(verify_len, tokens, uniforms, sa.B, sa.gamma, sa.V, GREEDY ? 1 : 0,
                               out_tokens, out_accept_len, sa.ws, L);
    const long long max_items = (long long)L.R * L.nch;
    const int grid = (int)std::min<long long>(sms, (max_items + kStatsWarps - 1) / kStatsWarps);
    if (g_ev_before) cudaEventRecord(g_ev_before, st);
    k_row_stats<ES, GREEDY><<<grid, kStatsWarps * 32, kStatsSmem, st>>>(sa, L);
    if (g_ev_after) cudaEventRecord(g_ev_after, st);
    k_accept<ES, GREEDY><<<sa.B, 128, 0, st>>>(aa, L);
    if (!GREEDY) {
        const long long items = (long long)sa.B * L.nch;
        k_resid_sum<ES><<<(unsigned)((items + 7) / 8), 256, 0, st>>>(ra, L);
        k_resid_pick<ES><<<(sa.B + 3) / 4, 128, 0, st>>>(ra, L);
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

    StatsArgs sa{(const char*)target_logits, (const char*)draft_logits, B, gamma, V, c_hi, c_lo,
                 (char*)workspace};
    AcceptArgs aa{(const char*)target_logits, (const char*)draft_logits, draft_tokens, uniforms,
                  out_tokens, out_accept_len, B, gamma, V, c_hi, c_lo, (char*)workspace};
    ResidArgs ra{(const char*)target_logits, (const char*)draft_logits, out_tokens, B, gamma, V,
                 c_hi, c_lo, (char*)workspace};
    cudaStream_t st = (cudaStream_t)stream;
    if (es == 2)
        return greedy ? launch_chain<2, true>(sa, aa, ra, verify_len, draft_tokens, uniforms, out_tokens,
                                              out_accept_len, L, sms, st)
                      : launch_chain<2, false>(sa, aa, ra, verify_len, draft_tokens, uniforms,
                                               out_tokens, out_accept_len, L, sms, st);
    return greedy ? launch_chain<4, true>(sa, aa, ra, verify_len, draft_tokens, uniforms, out_tokens,
                                          out_accept_len, L, sms, st)
                  : launch_chain<4, false>(sa, aa, ra, verify_len, draft_tokens, uniforms, out_tokens,
                                           out_accept_len, L, sms, st);
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
    return temperature == 0.0f ? 3 : 5;
}

}  // extern "C"
