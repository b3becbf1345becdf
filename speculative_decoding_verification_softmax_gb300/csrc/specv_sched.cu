// Confidence-scheduled verify lengths on GB300: one thread-block cluster per
// call for the batch schedulers, one warp per request for the static ones.
//
// Method (restated from the pages):
//   * Prefix survival s_{b,0} = 1, s_{b,k} = prod_{t<=k} c_{b,t} ("AngelSpec"
//     §4.2, eq. (20)) and estimated progress A_b(n) = sum_{k<=n} s_{b,k}
//     (eq. (21)).
//   * Candidates (b, k > min_len) ordered by survival, ties to the shallower
//     position then the lower request (top-K with shallow-first ties keeps
//     every request's kept drafts a contiguous prefix, §4.2).
//   * Budget N = sum_b (ell_b + 1) ("AngelSpec" §4.1): taking the first
//     N - B(min_len+1) candidates gives the best estimated progress tau(N) for
//     that budget; the call returns the allocation of the first N that
//     maximises tau(N) / C(N) (eq. (24) with every budget a candidate), or,
//     in Algorithm-1 mode ("UraionSpec" §3.5), stops at the first candidate
//     that does not strictly improve tau / C, or, in D-cut mode (§4.2,
//     eqs. (22)-(24)), takes the best of the ratio budgets.
//
// Numbers.  Survival products are fp64, left to right.  Each survival is then
// rounded to a multiple of 2^-46 and held as a 47-bit integer q: candidates
// are ordered by q, and progress values are exact 64-bit integer sums of q, so
// tau(N) does not depend on the order of summation and a parallel scan gives
// the same bits as a sequential sum.  Objectives tau / C are fp64 through
// explicit round-to-nearest intrinsics (no FMA contraction).
//
// GB300 has a narrow FP64 pipe, so the batch scheduler spreads its FP64 work
// (survival products, STS powers, objectives) over the CTAs of a cluster;
// the sort and the integer scan, which need no FP64, are repeated in every
// CTA so that no further exchange is needed.
#include <cooperative_groups.h>
#include <math.h>
#include <stdint.h>

#include "specv_common.cuh"
#include "specv_trace.h"

namespace cg = cooperative_groups;

namespace specv {

constexpr int kSchedThreads = 1024;
constexpr int kSchedMaxCluster = 16;
constexpr uint64_t kQField = (1ull << 47) - 1;  // survival field of a candidate key
constexpr int kRankMax = 4096;                  // candidates ordered by distributed ranking

struct SchedArgs {
    const float* conf;
    int32_t* out;
    int* status;
    int B, gamma, min_len, mode, nk, nc, npad;
    int has_sts;
    double kt[32];
    double kc[32];
    float sts[32];  // STS temperatures per position (has_sts)
};

// Confidence of position k (1-based), calibrated by c^(1/T_k) when STS
// temperatures are given ("UraionSpec" §2.4).
__device__ __forceinline__ double conf_at(const float* conf, const float* sts, int has_sts, size_t i, int k) {
    const double c = (double)conf[i];
    return has_sts ? pow(c, __ddiv_rn(1.0, (double)sts[k - 1])) : c;
}

// Survival s in [0, 1] as an integer multiple of 2^-46, rounded to nearest
// with ties to even.  Integer arithmetic on the bits of s: s = m * 2^(e-1075)
// with a 53-bit m, so s * 2^46 = m >> (1029 - e) plus the rounding of the
// bits shifted out (GB300's fp64 conversions are slow).
__device__ __forceinline__ uint64_t surv_q(double s) {
    const uint64_t bits = (uint64_t)__double_as_longlong(s);
    const int e = (int)(bits >> 52);
    if (e == 0) return 0;  // zero, or subnormal: far below 2^-47
    const uint64_t m = (bits & ((1ull << 52) - 1)) | (1ull << 52);
    const int sh = 1029 - e;  // >= 6 for s <= 1
    if (sh >= 54) return 0;   // s * 2^46 < 1/2
    const uint64_t q = m >> sh, rem = m & ((1ull << sh) - 1), half = 1ull << (sh - 1);
    return q + ((rem > half || (rem == half && (q & 1))) ? 1 : 0);
}

// Progress value t * 2^-46 of an integer sum of survivals: the double
// nearest to it (ties to even), built from the bits of t.
__device__ __forceinline__ double prog_value(uint64_t t) {
    if (t == 0) return 0.0;
    int ex = 63 - __clzll((long long)t);
    uint64_t m;
    if (ex <= 52) {
        m = t << (52 - ex);
    } else {
        const int sh = ex - 52;
        m = t >> sh;
        const uint64_t rem = t & ((1ull << sh) - 1), half = 1ull << (sh - 1);
        if (rem > half || (rem == half && (m & 1))) {
            ++m;
            if (m >> 53) {
                m >>= 1;
                ++ex;
            }
        }
    }
    return __longlong_as_double((long long)(((uint64_t)(ex - 46 + 1023) << 52) | (m & ((1ull << 52) - 1))));
}

// Candidate key, ascending = survival descending, then k, then b:
// [63:17] complement of q, [16:12] k - 1, [11:0] b.
__device__ __forceinline__ uint64_t cand_key(uint64_t q, int k, int b) {
    return ((kQField - q) << 17) | ((uint64_t)(k - 1) << 12) | (uint64_t)b;
}

__device__ __forceinline__ double cost_at(double N, const SchedArgs& a) {
    if (N <= a.kt[0]) return a.kc[0];
    if (N >= a.kt[a.nk - 1]) return a.kc[a.nk - 1];
    int i = 0;
    while (!(N < a.kt[i + 1])) ++i;
    return __dadd_rn(a.kc[i], __ddiv_rn(__dmul_rn(__dsub_rn(N, a.kt[i]), __dsub_rn(a.kc[i + 1], a.kc[i])),
                                        __dsub_rn(a.kt[i + 1], a.kt[i])));
}

// Bitonic compare-exchange stages with strides jmax..1 (all < 32) inside a warp.
__device__ __forceinline__ uint64_t warp_bitonic(uint64_t v, int i, int k, int jmax) {
    for (int j = jmax; j > 0; j >>= 1) {
        const uint64_t p = __shfl_xor_sync(0xffffffffu, v, j);
        const bool up = (i & k) == 0, low = (i & j) == 0;
        v = (up == low) ? (v < p ? v : p) : (v < p ? p : v);
    }
    return v;
}

// Largest value, ties to the smallest index (objectives are non-negative
// doubles, so their bit patterns order like their values).
__device__ __forceinline__ void warp_best(uint64_t& v, int& i) {
    for (int o = 16; o > 0; o >>= 1) {
        const uint64_t ov = __shfl_xor_sync(0xffffffffu, v, o);
        const int oi = __shfl_xor_sync(0xffffffffu, i, o);
        if (ov > v || (ov == v && oi < i)) {
            v = ov;
            i = oi;
        }
    }
}

__device__ __forceinline__ uint64_t obj_bits(double v) { return (uint64_t)__double_as_longlong(v); }

// Number of entries of the ascending array a[0, n) below x (n >= 1):
// branch-free binary search, the same trip count for every lane of a warp
// searching arrays of one length.
__device__ __forceinline__ int count_below(const uint64_t* a, int n, uint64_t x) {
    int lo = 0;
    for (int step = 1 << (31 - __clz(n)); step > 0; step >>= 1) {
        const int t = lo + step;
        if (t <= n && a[t - 1] < x) lo = t;
    }
    return lo;
}

// Split cluster barrier (PTX ISA, barrier.cluster): arrive without ordering
// memory, wait later.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }

// Outputs when there is nothing to schedule: every request invalid (bad
// confidence), or no candidates (min_len == gamma).
__device__ __forceinline__ void sched_trivial_out(const SchedArgs& a, bool bad, int tid) {
    for (int b = tid; b < a.B; b += blockDim.x) a.out[b] = bad ? -1 : a.min_len;
    if (bad && tid == 0) set_status(a.status, SPEC_ERR_CONFIDENCE);
}

__global__ void __launch_bounds__(kSchedThreads, 1) k_schedule(SchedArgs a) {
    cg::cluster_group cluster = cg::this_cluster();
    const int CL = (int)cluster.num_blocks();
    const int rank = (int)cluster.block_rank();
    extern __shared__ __align__(16) unsigned char smem_raw[];
    uint64_t* key = (uint64_t*)smem_raw;                 // [npad]: keys, then q, then tau; last: counts
    uint16_t* cb = (uint16_t*)(key + a.npad);            // [npad]: request of each sorted candidate
    double* stage = (double*)(cb + a.npad);              // [kSchedThreads]: confidences of one round
    uint64_t* kst = (uint64_t*)(stage + kSchedThreads);  // [kSchedThreads]: keys of one round
    // followed (nc <= kRankMax) by [npad] keys in rank order
    __shared__ unsigned long long s_base_local;
    __shared__ uint64_t s_base_part[kSchedMaxCluster];
    __shared__ uint64_t s_slot_v[kSchedMaxCluster];
    __shared__ int s_slot_i[kSchedMaxCluster];
    __shared__ uint64_t s_red_v[32];
    __shared__ int s_red_i[32];
    __shared__ int s_bad, s_npos, s_bestK, s_dcut_k;

    // (no early trigger of the next kernel here: placing the verification's
    // streaming CTAs on the other SMs while this cluster runs starts the 16
    // CTAs that must wait for this cluster's SMs late, and the streaming
    // pass's static split then ends late by as much)
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int B = a.B, G = a.gamma, ml = a.min_len, per = G - ml, nc = a.nc, npad = a.npad;
    // With STS the fp64 powers are split over the cluster and the keys are
    // exchanged; without, every CTA computes every survival itself (a few
    // fp64 products per request) and the cluster meets only at the end.
    const bool split = a.has_sts != 0;
    if (tid == 0) {
        s_bad = 0;
        s_base_local = 0;
        s_npos = 0;
    }
    if (!split) cluster_arrive_relaxed();  // waited on before the first store to another CTA
    __syncthreads();

    // the objective slice of this CTA: budgets K in [k_lo, k_lo + ccnt)
    // (exact scan and Algorithm 1); their round costs, one per thread while
    // the survival chains run, in csl[0 .. ccnt] (one past the slice for
    // Algorithm 1's look-ahead)
    const double N0 = __dmul_rn((double)B, (double)(ml + 1));
    const int cpc = (nc + 1 + CL - 1) / CL;
    const int k_lo = min(nc + 1, rank * cpc), ccnt = min(nc + 1, k_lo + cpc) - k_lo;
    double* csl = (double*)(kst + kSchedThreads + (nc <= kRankMax ? npad : 0));
    bool costs_done = a.mode == SPEC_SCHED_DCUT;
    uint64_t base = 0;
    if (split) {
        // every CTA checks the whole input, so that all take the same branch
        for (int i = tid; i < B * G; i += kSchedThreads) {
            const float c = a.conf[i];
            if (!(c >= 0.0f && c <= 1.0f)) s_bad = 1;
        }
        cluster.sync();  // also: every CTA runs before any shared-memory store across the cluster
        if (s_bad || nc == 0) {
            if (rank == 0) sched_trivial_out(a, s_bad != 0, tid);
            return;
        }
    }

    // 1. survivals in rounds of kSchedThreads / G requests: the round's
    //    (calibrated) confidences staged in shared memory by all threads, then
    //    one thread per request takes the products.  Split: this CTA's share
    //    of the requests, keys sent to every CTA; else all requests, checking
    //    the confidences on the way.
    {
        const int bpc = split ? (B + CL - 1) / CL : B;
        const int b_lo = min(B, rank * (split ? bpc : 0)), b_hi = min(B, b_lo + bpc);
        const int R = kSchedThreads / max(G, 1);
        costs_done = false;
        for (int r0 = b_lo; r0 < b_hi; r0 += R) {
            const int nr = min(R, b_hi - r0);
            if (tid < nr * G) {
                const int b = r0 + tid / G, k = tid - (tid / G) * G + 1;
                const size_t i = (size_t)b * G + k - 1;
                double c;
                if (split) {
                    c = conf_at(a.conf, a.sts, 1, i, k);
                } else {
                    const float cf = a.conf[i];
                    if (!(cf >= 0.0f && cf <= 1.0f)) s_bad = 1;
                    c = (cf >= 0.0f && cf <= 1.0f) ? (double)cf : 0.0;
                }
                stage[tid] = c;
            }
            __syncthreads();
            // the products, one thread per request, each survival written back
            // over its confidence (only the fp64 chain is sequential)
            if (tid < nr) {
                double* sr = stage + tid * G;
                double s = 1.0;
                for (int k = 0; k < G; ++k) {
                    s = __dmul_rn(s, sr[k]);
                    sr[k] = s;
                }
            } else if (!costs_done) {
                // meanwhile the idle threads take the round costs C(N0 + K)
                // of this CTA's objective slice (they do not depend on the order)
                for (int j = tid - nr; j <= ccnt; j += kSchedThreads - nr)
                    csl[j] = cost_at(__dadd_rn(N0, (double)(k_lo + j)), a);
            }
            costs_done = costs_done || nr < kSchedThreads;
            __syncthreads();
            // keys and the progress at min_len, one thread per (request, k)
            {
                uint64_t A = 0;
                if (tid < nr * G) {
                    const int j = tid / G, k = tid - j * G + 1, b = r0 + j;
                    const uint64_t q = surv_q(stage[tid]);
                    if (k <= ml)
                        A = q;
                    else
                        (split ? kst + j * per : key + (size_t)b * per)[k - ml - 1] = cand_key(q, k, b);
                }
                if (tid < nr) A += surv_q(1.0);  // the k = 0 term of request r0 + tid
                for (int o = 16; o > 0; o >>= 1) A += __shfl_xor_sync(0xffffffffu, A, o);
                if (lane == 0 && A) atomicAdd(&s_base_local, (unsigned long long)A);
            }
            __syncthreads();
            if (split) {
                const int nkeys = nr * per;  // candidate index of kst[j] is r0 * per + j
                for (int t = tid; t < nkeys * CL; t += kSchedThreads) {
                    const int j = t / CL, dst = t - j * CL;
                    *cluster.map_shared_rank(&key[r0 * per + j], dst) = kst[j];
                }
                __syncthreads();
            }
        }
    }
    for (int i = nc + tid; i < npad; i += kSchedThreads) key[i] = ~0ull;
    if (split) {
        if (tid < CL) *cluster.map_shared_rank(&s_base_part[rank], tid) = (uint64_t)s_base_local;
        cluster.sync();
        for (int r = 0; r < CL; ++r) base += s_base_part[r];
    } else {
        __syncthreads();
        if (s_bad || nc == 0) {
            cluster_wait();
            if (rank == 0) sched_trivial_out(a, s_bad != 0, tid);
            return;
        }
        base = s_base_local;
    }

    if (!costs_done) {
        for (int j = tid; j <= ccnt; j += kSchedThreads) csl[j] = cost_at(__dadd_rn(N0, (double)(k_lo + j)), a);
        __syncthreads();
    }
    if (!split) cluster_wait();  // every CTA of the cluster runs: stores across it follow

    // 2. order the candidates.  Up to kRankMax candidates, by rank: each
    //    request's keys already form an ascending run of `per`, so a key's rank
    //    is the sum over runs of the keys below it; every CTA ranks its share
    //    and stores the key at that rank in every CTA (one 64-bit store per
    //    CTA and candidate).  Above that, a bitonic network sorts the keys in
    //    every CTA.
    uint64_t* qv = key;  // keys in candidate order after this step, then their survivals q
    if (nc <= kRankMax) {
        uint64_t* sq = kst + kSchedThreads;  // [npad]
        for (int i = nc + tid; i < npad; i += kSchedThreads) sq[i] = 0;
        const int cpc = (nc + CL - 1) / CL, c_lo = min(nc, rank * cpc), c_hi = min(nc, c_lo + cpc);
        for (int i = c_lo + warp; i < c_hi; i += kSchedThreads / 32) {
            const uint64_t x = key[i];
            int below = 0;
            for (int r2 = lane; r2 < B; r2 += 32) below += count_below(key + r2 * per, per, x);
            for (int o = 16; o > 0; o >>= 1) below += __shfl_xor_sync(0xffffffffu, below, o);
            if (lane < CL) *cluster.map_shared_rank(&sq[below], lane) = x;
        }
        cluster.sync();
        qv = sq;
    } else {
        // bitonic: strides below 32 by warp shuffles, the others through
        // shared memory (npad >= 32, so the threads of a warp are all in or
        // all out)
        for (int i = tid; i < npad; i += kSchedThreads) {
            uint64_t v = key[i];
            for (int k = 2; k <= 32 && k <= npad; k <<= 1) v = warp_bitonic(v, i, k, k >> 1);
            key[i] = v;
        }
        __syncthreads();
        for (int k = 64; k <= npad; k <<= 1) {
            for (int j = k >> 1; j >= 32; j >>= 1) {
                for (int p = tid; p < (npad >> 1); p += kSchedThreads) {
                    const int i = ((p & ~(j - 1)) << 1) | (p & (j - 1));
                    const uint64_t x = key[i], y = key[i + j];
                    if ((x > y) == ((i & k) == 0)) {
                        key[i] = y;
                        key[i + j] = x;
                    }
                }
                __syncthreads();
            }
            for (int i = tid; i < npad; i += kSchedThreads) key[i] = warp_bitonic(key[i], i, k, 16);
            __syncthreads();
        }
    }

    // 3. survivals q in sorted order from the sorted keys, the request of
    //    each, and the count of positive ones (a prefix, q being descending)
    int npos = 0;
    for (int i = tid; i < npad; i += kSchedThreads) {
        const uint64_t kk = qv[i];
        uint64_t q = 0;
        if (i < nc) {
            q = kQField - (kk >> 17);
            cb[i] = (uint16_t)(kk & 4095u);
        }
        qv[i] = q;
        npos += q > 0;
    }
    for (int o = 16; o > 0; o >>= 1) npos += __shfl_xor_sync(0xffffffffu, npos, o);
    if (lane == 0 && npos) atomicAdd(&s_npos, npos);
    __syncthreads();

    // 4. tau(K) = base + q_0 + ... + q_{K-1}, exact, in key[K-1]: each thread
    //    scans a contiguous segment; segment totals by warp and block scans
    {
        const int E = npad > kSchedThreads ? npad / kSchedThreads : 1;
        const bool has = tid * E < npad;
        uint64_t run = 0;
        if (has)
            for (int e = 0; e < E; ++e) run += qv[tid * E + e];
        uint64_t incl = run;
        for (int o = 1; o < 32; o <<= 1) {
            const uint64_t t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        if (lane == 31) s_red_v[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const uint64_t w = s_red_v[lane];
            uint64_t wi = w;
            for (int o = 1; o < 32; o <<= 1) {
                const uint64_t t = __shfl_up_sync(0xffffffffu, wi, o);
                if (lane >= o) wi += t;
            }
            s_red_v[lane] = wi - w;
        }
        __syncthreads();
        uint64_t off = base + s_red_v[warp] + (incl - run);
        if (has)
            for (int e = 0; e < E; ++e) {
                off += qv[tid * E + e];
                key[tid * E + e] = off;
            }
        __syncthreads();
    }

    // 5. objectives, split over the cluster (costs of the slice from csl)
    auto tau_at = [&](int K) -> double { return prog_value(K == 0 ? base : key[K - 1]); };
    auto obj_at = [&](int K) -> double { return __ddiv_rn(tau_at(K), csl[K - k_lo]); };
    const int k_hi = k_lo + ccnt;
    uint64_t bv = 0;
    int bi = 0x7fffffff;
    if (a.mode == SPEC_SCHED_EXACT) {
        for (int K = k_lo + tid; K < k_hi; K += kSchedThreads) {
            const uint64_t v = obj_bits(obj_at(K));
            if (v > bv || (v == bv && K < bi)) {
                bv = v;
                bi = K;
            }
        }
    } else if (a.mode == SPEC_SCHED_ALGORITHM1) {
        // the first valid candidate i (i < npos) that does not strictly
        // improve tau / C, over this CTA's slice
        const int i_hi = min(s_npos, k_hi);
        for (int i = k_lo + tid; i < i_hi; i += kSchedThreads)
            if (!(obj_at(i + 1) > obj_at(i)) && i < bi) bi = i;
    } else if (rank == 0 && warp == 0) {
        // D-cut: K_i = max(N0, ceil(rho_i * B(gamma+1))) for the nk ratios
        const double Nmax = __dmul_rn((double)B, (double)(G + 1));
        int take = 0;
        if (lane < a.nk) {
            double K = ceil(__dmul_rn(a.kt[lane], Nmax));
            if (K < N0) K = N0;
            if (K > Nmax) K = Nmax;
            take = (int)__dsub_rn(K, N0);
            bv = obj_bits(__ddiv_rn(tau_at(take), a.kc[lane]));
            bi = lane;
        }
        warp_best(bv, bi);
        const int take_best = __shfl_sync(0xffffffffu, take, bi & 31);
        if (lane == 0) s_dcut_k = take_best;
    }
    if (a.mode != SPEC_SCHED_DCUT) {
        if (a.mode == SPEC_SCHED_EXACT) {
            warp_best(bv, bi);
        } else {
            for (int o = 16; o > 0; o >>= 1) bi = min(bi, __shfl_xor_sync(0xffffffffu, bi, o));
        }
        if (lane == 0) {
            s_red_v[warp] = bv;
            s_red_i[warp] = bi;
        }
        __syncthreads();
        if (warp == 0) {
            bv = s_red_v[lane];
            bi = s_red_i[lane];
            if (a.mode == SPEC_SCHED_EXACT) {
                warp_best(bv, bi);
            } else {
                for (int o = 16; o > 0; o >>= 1) bi = min(bi, __shfl_xor_sync(0xffffffffu, bi, o));
            }
            if (lane == 0) {
                *cluster.map_shared_rank(&s_slot_v[rank], 0) = bv;
                *cluster.map_shared_rank(&s_slot_i[rank], 0) = bi;
            }
        }
    }
    cluster.sync();
    if (rank != 0) return;

    // 6. rank 0: the chosen budget and the per-request counts
    if (tid == 0) {
        int bestK;
        if (a.mode == SPEC_SCHED_DCUT) {
            bestK = s_dcut_k;
        } else if (a.mode == SPEC_SCHED_EXACT) {
            uint64_t v = s_slot_v[0];
            int k = s_slot_i[0];
            for (int r = 1; r < CL; ++r)
                if (s_slot_v[r] > v || (s_slot_v[r] == v && s_slot_i[r] < k)) {
                    v = s_slot_v[r];
                    k = s_slot_i[r];
                }
            bestK = k;
        } else {
            int k = s_npos;
            for (int r = 0; r < CL; ++r) k = min(k, s_slot_i[r]);
            bestK = k;
        }
        s_bestK = bestK;
    }
    __syncthreads();
    const int bestK = s_bestK;
    int* count = (int*)key;  // tau is no longer needed
    for (int b = tid; b < B; b += kSchedThreads) count[b] = 0;
    __syncthreads();
    for (int i = tid; i < bestK; i += kSchedThreads) atomicAdd(&count[cb[i]], 1);
    __syncthreads();
    for (int b = tid; b < B; b += kSchedThreads) a.out[b] = ml + count[b];
}

// Static verify lengths: the leading positions whose (calibrated) confidence
// is at least the threshold, clamped to [min_len, max_len].  One warp per
// request, one lane per position; one warp per CTA spreads the fp64 powers of
// STS over the SMs.
__global__ void __launch_bounds__(32) k_schedule_static(const float* conf, int G, double threshold, int max_len,
                                                        int min_len, int has_sts, SchedArgs sa, int32_t* out,
                                                        int* status) {
    pdl_trigger();  // the next kernel may be placed now (it waits for these results)
    const int b = blockIdx.x, lane = threadIdx.x;
    bool bad = false, ok = true;
    if (conf && lane < G) {
        const float c = conf[(size_t)b * G + lane];
        bad = !(c >= 0.0f && c <= 1.0f);
        if (!bad && threshold > 0.0) ok = conf_at(conf, sa.sts, has_sts, (size_t)b * G + lane, lane + 1) >= threshold;
    }
    const unsigned badm = __ballot_sync(0xffffffffu, bad);
    const unsigned okm = __ballot_sync(0xffffffffu, ok);
    if (lane == 0) {
        if (badm) {
            out[b] = -1;
            set_status(status, SPEC_ERR_CONFIDENCE);
            return;
        }
        int n = ~okm ? __ffs(~okm) - 1 : 32;
        n = n < max_len ? n : max_len;
        out[b] = n < min_len ? min_len : n;
    }
}

}  // namespace specv

using namespace specv;

namespace {

// Dynamic shared memory of k_schedule for a padded candidate count (the
// ranked path keeps the survivals in rank order in a second array).
size_t sched_smem_bytes(int npad, int nc, int cl) {
    const size_t cpc = (size_t)(nc + 1 + cl - 1) / cl;
    return (size_t)npad * 10 + (size_t)kSchedThreads * 16 + 16 + (nc <= kRankMax ? (size_t)npad * 8 : 0) +
           (cpc + 1) * 8;
}

// Cluster size of k_schedule per device: 16 CTAs where the GPU can place such
// a cluster at the largest shared-memory size, else the portable 8; 0 = not
// set up yet.
int g_sched_cluster[64];

int sched_cluster_size(int dev) {
    if (g_sched_cluster[dev]) return g_sched_cluster[dev];
    int npad_max = 32;
    while (npad_max < SPEC_MAX_SCHED_CANDIDATES) npad_max <<= 1;
    const size_t smem_max = sched_smem_bytes(npad_max, SPEC_MAX_SCHED_CANDIDATES, 8);
    if (cudaFuncSetAttribute((const void*)k_schedule, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem_max) != cudaSuccess)
        return 0;
    int cl = 8;
    if (cudaFuncSetAttribute((const void*)k_schedule, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
        cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(kSchedMaxCluster);
        cfg.blockDim = dim3(kSchedThreads);
        cfg.dynamicSmemBytes = smem_max;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = kSchedMaxCluster;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, (const void*)k_schedule, &cfg) == cudaSuccess && n > 0)
            cl = kSchedMaxCluster;
        else
            cudaGetLastError();
    } else {
        cudaGetLastError();
    }
    g_sched_cluster[dev] = cl;
    return cl;
}

}  // namespace

extern "C" {

size_t spec_schedule_workspace_bytes(int B, int gamma) {
    if (B < 0 || B > SPEC_MAX_BATCH || gamma < 0 || gamma > SPEC_MAX_GAMMA) return 0;
    return 256;
}

static bool sts_ok(const float* T, int gamma) {
    if (!T) return true;
    for (int k = 0; k < gamma; ++k)
        if (!(T[k] > 0.0f) || !isfinite(T[k])) return false;
    return true;
}

int spec_schedule(const float* confidence, int B, int gamma, const spec_cost_table* cost, int min_len,
                  spec_sched_mode mode, const float* sts_temperature, int32_t* out_verify_len, void* workspace,
                  size_t workspace_bytes, spec_stream_t stream) {
    TraceRange tr("spec_schedule");
    if (B < 0 || B > SPEC_MAX_BATCH || gamma < 0 || gamma > SPEC_MAX_GAMMA || min_len < 0 || min_len > gamma)
        return SPEC_ERR_SHAPE;
    if ((long long)B * (gamma - min_len) > SPEC_MAX_SCHED_CANDIDATES) return SPEC_ERR_SHAPE;
    if (mode != SPEC_SCHED_EXACT && mode != SPEC_SCHED_ALGORITHM1 && mode != SPEC_SCHED_DCUT) return SPEC_ERR_SHAPE;
    if (!cost) return SPEC_ERR_NULL;
    if (cost->n < 1 || cost->n > 32) return SPEC_ERR_COST_TABLE;
    for (int i = 0; i < cost->n; ++i) {
        if (!isfinite(cost->tokens[i]) || !isfinite(cost->cost_ms[i]) || !(cost->cost_ms[i] > 0.0))
            return SPEC_ERR_COST_TABLE;
        if (i > 0 && !(cost->tokens[i] > cost->tokens[i - 1])) return SPEC_ERR_COST_TABLE;
        if (mode == SPEC_SCHED_DCUT && !(cost->tokens[i] > 0.0 && cost->tokens[i] <= 1.0)) return SPEC_ERR_COST_TABLE;
    }
    if (!sts_ok(sts_temperature, gamma)) return SPEC_ERR_SHAPE;
    if (B == 0) return SPEC_OK;
    if (!out_verify_len || !workspace || (gamma > 0 && !confidence)) return SPEC_ERR_NULL;
    if (((uintptr_t)out_verify_len & 3) || ((uintptr_t)workspace & 15) || ((uintptr_t)confidence & 3))
        return SPEC_ERR_ALIGN;
    if (workspace_bytes < 256) return SPEC_ERR_WORKSPACE;

    SchedArgs a;
    a.conf = confidence;
    a.out = out_verify_len;
    a.status = (int*)workspace;
    a.B = B;
    a.gamma = gamma;
    a.min_len = min_len;
    a.mode = (int)mode;
    a.nk = cost->n;
    a.nc = B * (gamma - min_len);
    int npad = 32;  // a power of two, at least one warp
    while (npad < a.nc) npad <<= 1;
    a.npad = npad;
    for (int i = 0; i < 32; ++i) {
        a.kt[i] = i < cost->n ? cost->tokens[i] : 0.0;
        a.kc[i] = i < cost->n ? cost->cost_ms[i] : 0.0;
        a.sts[i] = (sts_temperature && i < gamma) ? sts_temperature[i] : 1.0f;
    }
    a.has_sts = sts_temperature ? 1 : 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SPEC_ERR_CUDA;
    const int cl = sched_cluster_size(dev);
    if (!cl) return SPEC_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cl);
    cfg.blockDim = dim3(kSchedThreads);
    cfg.dynamicSmemBytes = sched_smem_bytes(npad, a.nc, cl);
    cfg.stream = (cudaStream_t)stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, k_schedule, a) != cudaSuccess) return SPEC_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

int spec_schedule_static(const float* confidence, int B, int gamma, float threshold, int max_len, int min_len,
                         const float* sts_temperature, int32_t* out_verify_len, void* workspace,
                         size_t workspace_bytes, spec_stream_t stream) {
    TraceRange tr("spec_schedule_static");
    if (B < 0 || B > SPEC_MAX_BATCH || gamma < 0 || gamma > SPEC_MAX_GAMMA || min_len < 0 || min_len > max_len ||
        max_len > gamma)
        return SPEC_ERR_SHAPE;
    if (!(threshold == threshold)) return SPEC_ERR_SHAPE;
    if (!sts_ok(sts_temperature, gamma)) return SPEC_ERR_SHAPE;
    if (B == 0) return SPEC_OK;
    if (!out_verify_len || !workspace || (threshold > 0.0f && gamma > 0 && !confidence)) return SPEC_ERR_NULL;
    if (((uintptr_t)out_verify_len & 3) || ((uintptr_t)workspace & 15) || ((uintptr_t)confidence & 3))
        return SPEC_ERR_ALIGN;
    if (workspace_bytes < 256) return SPEC_ERR_WORKSPACE;
    SchedArgs sa;
    for (int i = 0; i < 32; ++i) sa.sts[i] = (sts_temperature && i < gamma) ? sts_temperature[i] : 1.0f;
    k_schedule_static<<<B, 32, 0, (cudaStream_t)stream>>>(gamma > 0 ? confidence : nullptr, gamma,
                                                           (double)threshold, max_len, min_len,
                                                           sts_temperature ? 1 : 0, sa, out_verify_len,
                                                           (int*)workspace);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // extern "C"
