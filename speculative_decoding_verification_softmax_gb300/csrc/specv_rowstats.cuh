// Row statistics: the HBM-streaming pass of batched verification.
//
// For every needed logit row (target rows 0..ell_b, and at T > 0 draft rows
// 0..ell_b-1 of request b) and every 4 KiB chunk of it, one warp computes
//   T > 0 : Mc = ceil(max_v z_v * c) (an integer-valued scale) and
//           S_c = sum_v 2^(z_v * c - Mc), c = log2(e) / T carried as c_hi + c_lo,
//   T == 0: the chunk max and the lowest index attaining it,
// i.e. the per-chunk pieces of the temperature softmax normaliser ("UraionSpec",
// §2.1, eq. (acceptance) is stated on p = softmax(z / T)) or of the greedy
// argmax.  The accept kernel merges the chunks of a row exactly (power-of-two
// rescaling).
//
// Layout: a persistent grid, one CTA per SM, 20 warps.  Each warp owns a ring
// of kStages shared-memory stages that it fills itself with 1-D bulk copies
// (cp.async.bulk, completion on an mbarrier) and consumes in order; no
// cross-warp synchronisation.  Work items (compact row, chunk) are dealt to
// warps round-robin; rows are listed request by request.
//
// Two variants:
//   ALIGNED  every row starts on a 16-byte boundary (16-byte aligned bases and
//            V * element size a multiple of 16): whole chunks are copied, the
//            cursor is advanced uniformly by all lanes, rows come from a table
//            in shared memory.
//   general  rows may start anywhere (element-aligned): the aligned interior
//            of each chunk is copied and up to 15 head / 7 tail elements are
//            loaded by lanes; per-stage descriptors live in shared memory.
#pragma once

#include "specv_common.cuh"

namespace specv {

// Descriptor of the chunk that occupies one ring stage (general variant).
struct StageDesc {
    ChunkSpan sp;
    int g;  // global row id: target rows [0, B(gamma+1)), then draft rows
    int c;  // chunk index within the row
};

constexpr int kStatsThreads = kStatsWarps * 32;
constexpr int kTableRows = 4096;  // compact rows listed in shared memory (more: prefix walk)
constexpr size_t kRingBytes = (size_t)kStatsWarps * kStages * kChunkBytes;
constexpr size_t kBarBytes = (size_t)kStatsWarps * kStages * 8;
constexpr size_t kDescBytes = (size_t)kStatsWarps * kStages * sizeof(StageDesc);
constexpr size_t kPrefixBytes = (SPEC_MAX_BATCH + 1) * 4;
constexpr size_t kStatsSmem = kRingBytes + kBarBytes + kDescBytes + kPrefixBytes + kTableRows * 4 + 128;
// the packed layout keeps each compact row's packed row index beside the table
constexpr size_t kStatsSmemPacked = kStatsSmem + kTableRows * 4;
constexpr int kVecPerLane = kChunkBytes / 16 / 32;  // 16-byte vectors per lane in one chunk

struct StatsArgs {
    const char* target;
    const char* draft;
    const int32_t* verify_len;
    int B, gamma, V;
    float c_hi, c_lo;
    char* ws;
    RowMap rm;
    int expire_first;  // test hook: each warp's first wait counts as expired (0 in normal use)
};

// Rows a request needs: target 0..ell and (T > 0) draft 0..ell-1; 0 when
// verify_len is out of range or packed rows fall outside the packed arrays
// (the finish kernel marks the request invalid).
template <bool GREEDY, bool PACKED>
__device__ __forceinline__ int rows_of(const int32_t* verify_len, const RowMap& rm, int b, int gamma) {
    const int ell = verify_len ? verify_len[b] : gamma;
    if (ell < 0 || ell > gamma) return 0;
    if (PACKED && !rows_in_range(rm, b, ell, !GREEDY)) return 0;
    return GREEDY ? ell + 1 : 2 * ell + 1;
}

// Global row id of row k of request b (which needs cnt rows).
template <bool GREEDY>
__device__ __forceinline__ int row_id(int b, int k, int cnt, int gamma, int T1) {
    const int ell = GREEDY ? cnt - 1 : (cnt - 1) >> 1;
    return k <= ell ? b * (gamma + 1) + k : T1 + b * gamma + (k - ell - 1);
}

// prefix[b] = rows of requests < b, prefix[B] = total.  Whole CTA; ends
// with a barrier, so every thread sees the prefix.
template <bool GREEDY, bool PACKED>
__device__ void block_row_prefix(const int32_t* verify_len, const RowMap& rm, int B, int gamma, int* prefix) {
    __shared__ int s_w[32];
    __shared__ int s_total;
    constexpr int PER = (SPEC_MAX_BATCH + kStatsThreads - 1) / kStatsThreads;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int cnt[PER];
    int mine = 0;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int b = tid * PER + i;
        cnt[i] = b < B ? rows_of<GREEDY, PACKED>(verify_len, rm, b, gamma) : 0;
        mine += cnt[i];
    }
    int incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) s_w[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int w = lane < kStatsWarps ? s_w[lane] : 0;
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += v;
        }
        s_w[lane] = wi - w;
        if (lane == 31) s_total = wi;
    }
    __syncthreads();
    int off = s_w[warp] + incl - mine;
    const int total = s_total;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int b = tid * PER + i;
        if (b < B) prefix[b] = off;
        off += cnt[i];
    }
    if (tid == 0) prefix[B] = total;
    __syncthreads();
}

// table[r] = global row id of compact row r (when the total fits), and for
// the packed layout ptable[r] = its row in the packed target or draft array:
// one warp per request writes its rows.  No barrier inside.
template <bool GREEDY, bool PACKED>
__device__ void block_row_table(const int* prefix, int B, int gamma, const RowMap& rm, int* table, int* ptable) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int T1 = B * (gamma + 1);
    for (int b = warp; b < B; b += kStatsWarps) {
        const int p0 = prefix[b], cnt = prefix[b + 1] - p0;
        if (cnt == 0) continue;
        const int ell = GREEDY ? cnt - 1 : (cnt - 1) >> 1;
        const int t0 = PACKED ? rm.trow[b] : 0;
        const int d0 = (PACKED && !GREEDY && ell > 0) ? rm.drow[b] : 0;
        for (int k = lane; k < cnt; k += 32) {
            table[p0 + k] = row_id<GREEDY>(b, k, cnt, gamma, T1);
            if (PACKED) ptable[p0 + k] = k <= ell ? t0 + k : d0 + (k - ell - 1);
        }
    }
}

// The request owning compact row r: the largest b with prefix[b] <= r.
__device__ __forceinline__ int request_of_row(const int* prefix, int B, int r) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (prefix[mid] <= r) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// Statistics of one chunk: nvec 16-byte vectors in shared memory holding the
// elements [base, base + nvec * 16 / ES), plus (general variant) one scalar
// element per lane (si >= 0).
template <int ES, bool GREEDY, int NVEC>
__device__ __forceinline__ float2 chunk_stats(const uint4* sm, int nvec_rt, int base, int si, float sv, int lane,
                                              float c_hi, float c_lo) {
    constexpr int EPV = 16 / ES;  // elements per 16-byte vector
    const int nvec = NVEC > 0 ? NVEC : nvec_rt;  // NVEC > 0: a full chunk, loops unroll completely

    if (GREEDY) {
        // One pass: each lane's max and the first of its vectors attaining it
        // (strict >, lanes walk their vectors in increasing index order).
        float lm = -INFINITY;
        int lv = lane;  // stays at the lane's first vector if all its values are -inf
        bool nan = false;
        for (int i = lane; i < nvec; i += 32) {
            float vf;
            if (ES == 2) {
                const uint4 x = sm[i];
                const uint32_t vm = bf16x2_max_nan(bf16x2_max_nan(x.x, x.y), bf16x2_max_nan(x.z, x.w));
                vf = fmax_nan(bf16_lo(vm), bf16_hi(vm));
            } else {
                const float4 x = ((const float4*)sm)[i];
                vf = fmax_nan(fmax_nan(x.x, x.y), fmax_nan(x.z, x.w));
            }
            nan |= vf != vf;
            if (vf > lm) {
                lm = vf;
                lv = i;
            }
        }
        if (si >= 0) nan |= sv != sv;
        nan = __any_sync(0xffffffffu, nan);
        float m = fmax_nan(lm, si >= 0 ? sv : -INFINITY);
        m = nan ? __int_as_float(0x7fc00000) : warp_max_nan(m);
        int best = 0x7fffffff;
        if (!nan) {
            if (lv < nvec && lm == m) {
                // the lowest index equal to m inside the lane's first maximal vector
                const int b0 = base + lv * EPV;
                if (ES == 2) {
                    const uint4 x = sm[lv];
                    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                    for (int k = 3; k >= 0; --k) {
                        if (bf16_hi(w[k]) == m) best = b0 + 2 * k + 1;
                        if (bf16_lo(w[k]) == m) best = b0 + 2 * k;
                    }
                } else {
                    const float4 x = ((const float4*)sm)[lv];
                    const float w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                    for (int k = 3; k >= 0; --k)
                        if (w[k] == m) best = b0 + k;
                }
            }
            if (si >= 0 && sv == m) best = min(best, si);
        }
        best = warp_min_i(best);
        return make_float2(m, __int_as_float(best));
    }

    // pass 1: max (NaN-propagating)
    float m;
    if (ES == 2) {
        uint32_t pm = 0xFF80FF80u;  // (-inf, -inf)
        int i = lane;
        for (; i + 32 < nvec; i += 64) {
            const uint4 x = sm[i], y = sm[i + 32];
            pm = bf16x2_max_nan(pm, bf16x2_max_nan(bf16x2_max_nan(x.x, x.y), bf16x2_max_nan(x.z, x.w)));
            pm = bf16x2_max_nan(pm, bf16x2_max_nan(bf16x2_max_nan(y.x, y.y), bf16x2_max_nan(y.z, y.w)));
        }
        if (i < nvec) {
            const uint4 x = sm[i];
            pm = bf16x2_max_nan(pm, bf16x2_max_nan(bf16x2_max_nan(x.x, x.y), bf16x2_max_nan(x.z, x.w)));
        }
        m = fmax_nan(bf16_lo(pm), bf16_hi(pm));
    } else {
        m = -INFINITY;
        for (int i = lane; i < nvec; i += 32) {
            const float4 x = ((const float4*)sm)[i];
            m = fmax_nan(m, fmax_nan(fmax_nan(x.x, x.y), fmax_nan(x.z, x.w)));
        }
    }
    if (si >= 0) m = fmax_nan(m, sv);
    m = warp_max_nan(m);

    // T > 0: sum of 2^(z*c - Mc) with the integer scale Mc = ceil(max * c)
    if (m != m || m == INFINITY) return make_float2(__int_as_float(0x7fc00000), 0.f);
    if (m == -INFINITY) return make_float2(-INFINITY, 0.f);
    const float Mc = ceilf(fmaf(m, c_hi, m * c_lo));
    // |max| * log2(e) / T beyond the fp32 range: no usable scale, reported
    // like a non-finite row
    if (!(fabsf(Mc) <= 3.0e38f)) return make_float2(__int_as_float(0x7fc00000), 0.f);
    // packed FP32x2 arithmetic: (z*c_hi - Mc) + z*c_lo for two elements per FMA
    const float2 ch2 = make_float2(c_hi, c_hi), cl2 = make_float2(c_lo, c_lo), nm2 = make_float2(-Mc, -Mc);
    float2 p0 = make_float2(0.f, 0.f), p1 = p0;
    auto pair = [&](float z0, float z1) -> float2 {
        const float2 z = make_float2(z0, z1);
        const float2 t = __ffma2_rn(z, cl2, __ffma2_rn(z, ch2, nm2));
        return make_float2(ex2_approx(t.x), ex2_approx(t.y));
    };
    if (ES == 2) {
#pragma unroll 4
        for (int i = lane; i < nvec; i += 32) {
            const uint4 x = sm[i];
            p0 = __fadd2_rn(p0, pair(bf16_lo(x.x), bf16_hi(x.x)));
            p1 = __fadd2_rn(p1, pair(bf16_lo(x.y), bf16_hi(x.y)));
            p0 = __fadd2_rn(p0, pair(bf16_lo(x.z), bf16_hi(x.z)));
            p1 = __fadd2_rn(p1, pair(bf16_lo(x.w), bf16_hi(x.w)));
        }
    } else {
#pragma unroll 4
        for (int i = lane; i < nvec; i += 32) {
            const float4 x = ((const float4*)sm)[i];
            p0 = __fadd2_rn(p0, pair(x.x, x.y));
            p1 = __fadd2_rn(p1, pair(x.z, x.w));
        }
    }
    float a0 = p0.x, a1 = p0.y, a2 = p1.x, a3 = p1.y;
    if (si >= 0) a0 += scaled_exp(sv, c_hi, c_lo, Mc);
    return make_float2(Mc, warp_sum((a0 + a1) + (a2 + a3)));
}

// PACKED: rows addressed through the row index of a packed layout (the
// padded layout's kernels carry none of that code).
template <int ES, bool GREEDY, bool ALIGNED, bool PACKED>
__global__ void __launch_bounds__(kStatsThreads, 1) k_row_stats(StatsArgs a, Layout L) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = (unsigned char*)(((uintptr_t)smem_raw + 127) & ~uintptr_t(127));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    unsigned char* ring = smem + (size_t)warp * kStages * kChunkBytes;
    uint64_t* bars = (uint64_t*)(smem + kRingBytes) + warp * kStages;
    StageDesc* desc = (StageDesc*)(smem + kRingBytes + kBarBytes) + warp * kStages;
    int* prefix = (int*)(smem + kRingBytes + kBarBytes + kDescBytes);
    int* table = prefix + (SPEC_MAX_BATCH + 1);
    int* ptable = table + kTableRows;  // packed layout only (in its larger allocation)
    int* hdr = (int*)(a.ws + L.hdr);
    float2* partial = (float2*)(a.ws + L.partial);
    __shared__ int s_exited, s_failed;  // warps done / any wait expired (this CTA)

    if (lane == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    if (tid == 0) s_exited = s_failed = 0;  // published by the barriers in block_row_prefix
    // launched as a programmatic dependent of the preceding kernel in the
    // stream: nothing in global memory is read or written before its results
    // are complete and visible
    pdl_wait();
    if (blockIdx.x == 0 && tid == 0) {  // per-call reset of the status words (only the
        hdr[kHdrStatus] = 0;             // finish kernel, which runs after every CTA of
        hdr[kHdrEvents] = 0;             // this grid, sets them)
    }
    block_row_prefix<GREEDY, PACKED>(a.verify_len, a.rm, a.B, a.gamma, prefix);
    pdl_trigger();

    const int nch = L.nch;
    const int n_rows = prefix[a.B];
    const long long total = (long long)n_rows * nch;
    const int W = gridDim.x * kStatsWarps;
    // warps numbered across the grid (local warp index major), so that the
    // items left over by W not dividing the total spread over every SM
    const int gw = warp * gridDim.x + blockIdx.x;
    const bool has_items = gw < total;
    const long long count = has_items ? (total - gw + W - 1) / W : 0;  // items of this warp
    const int Wq = W / nch, Wr = W - Wq * nch;
    const int T1 = a.B * (a.gamma + 1);
    // the row table pays off only when warps take more items than the first
    // kStages (issued from the prefix before the table could exist)
    const bool use_table = n_rows <= kTableRows && total > (long long)W * kStages;
    bool table_ready = false;  // the first copies are issued before the table is built

    // A cursor over this warp's items: (compact row, chunk) and the request
    // of the row (for the prefix walk when the table does not fit).
    struct Cursor {
        int r, c, b;
    };
    auto advance = [&](Cursor& k) {
        k.c += Wr;
        k.r += Wq;
        if (k.c >= nch) {
            k.c -= nch;
            ++k.r;
        }
    };
    auto row_of = [&](Cursor& k) -> int {
        if (table_ready) return table[k.r];
        while (prefix[k.b + 1] <= k.r) ++k.b;
        const int cnt = prefix[k.b + 1] - prefix[k.b];
        return row_id<GREEDY>(k.b, k.r - prefix[k.b], cnt, a.gamma, T1);
    };
    auto row_ptr = [&](const Cursor& k, int g) -> const char* {
        if constexpr (!PACKED) return g < T1 ? a.target + (size_t)g * a.V * ES : a.draft + (size_t)(g - T1) * a.V * ES;
        if (table_ready) return (g < T1 ? a.target : a.draft) + (size_t)ptable[k.r] * a.V * ES;
        if (g < T1) {
            const int b = g / (a.gamma + 1);
            return a.target + target_row(a.rm, b, g - b * (a.gamma + 1), a.gamma + 1) * a.V * ES;
        }
        const int gd = g - T1, b = gd / a.gamma;
        return a.draft + draft_row(a.rm, b, gd - b * a.gamma, a.gamma) * a.V * ES;
    };

    // Every warp ends here: the last warp of the CTA to leave writes the CTA's
    // word (SPEC_ERR_TIMEOUT if any of its waits expired, else SPEC_OK).
    auto warp_exit = [&](bool failed) {
        if (lane == 0) {
            if (failed) atomicOr(&s_failed, 1);
            __threadfence_block();
            if (atomicAdd(&s_exited, 1) == kStatsWarps - 1) {
                __threadfence_block();
                ((int*)(a.ws + L.ctaw))[blockIdx.x] = atomicOr(&s_failed, 0) ? SPEC_ERR_TIMEOUT : SPEC_OK;
            }
        }
    };

    Cursor ic{gw / nch, gw - (gw / nch) * nch, 0};  // issue cursor
    if (has_items) ic.b = request_of_row(prefix, a.B, ic.r);
    Cursor cc = ic;  // consume cursor
    uint32_t pending = 0;  // bit s: a copy is in flight on stage s
    uint32_t phase = 0;    // bit s: parity of the next wait on stage s
    long long issued = 0;

    // Issue the copy of the item under the issue cursor into stage s.
    auto issue = [&](int s) {
        const int g = row_of(ic);
        const char* rowp = row_ptr(ic, g);
        const int e0 = ic.c * L.CH, e1 = min(a.V, e0 + L.CH);
        bool copy;
        const char* src;
        uint32_t bytes;
        if constexpr (ALIGNED) {
            copy = true;
            src = rowp + (size_t)e0 * ES;
            bytes = (uint32_t)((e1 - e0) * ES);
        } else {
            StageDesc d;
            d.sp = chunk_span<ES>(rowp, e0, e1);
            d.g = g;
            d.c = ic.c;
            if (lane == 0) desc[s] = d;
            copy = d.sp.ia < d.sp.ib;
            src = rowp + (size_t)d.sp.ia * ES;
            bytes = (uint32_t)((d.sp.ib - d.sp.ia) * ES);
        }
        if (copy) {
            if (lane == 0) {
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(&bars[s], bytes);
                bulk_g2s(ring + (size_t)s * kChunkBytes, src, bytes, &bars[s]);
            }
            pending |= 1u << s;
        }
        advance(ic);
        ++issued;
    };

#pragma unroll 1
    for (int s = 0; s < kStages && issued < count; ++s) issue(s);
    // the row table is built while those copies are in flight
    if (use_table) {
        block_row_table<GREEDY, PACKED>(prefix, a.B, a.gamma, a.rm, table, ptable);
        __syncthreads();
        table_ready = true;
    }
    if (!has_items) {
        warp_exit(false);
        return;
    }
    __syncwarp();

    int s = 0;
    bool failed = false;
#pragma unroll 1
    for (long long done = 0; done < count; ++done) {
        int g, c, nvec, base, si = -1;
        float sv = 0.f;
        if constexpr (ALIGNED) {
            g = row_of(cc);
            c = cc.c;
            base = c * L.CH;
            nvec = (min(a.V, base + L.CH) - base) * ES / 16;
        } else {
            const StageDesc d = desc[s];
            g = d.g;
            c = d.c;
            base = d.sp.ia;
            nvec = (d.sp.ib - d.sp.ia) * ES / 16;
            si = span_scalar_index(d.sp, lane);
            if (si >= 0) sv = load_logit<ES>(d.sp.rowp, si);
        }
        if (pending & (1u << s)) {
            // every lane waits (each observes the copy's completion); the warp
            // goes on only if all of them saw it
            const bool ok = !(a.expire_first && done == 0) && mbar_wait_bounded(&bars[s], (phase >> s) & 1u);
            if (!__all_sync(0xffffffffu, ok)) {
                failed = true;
                break;
            }
            phase ^= 1u << s;
            pending &= ~(1u << s);
        }
        const uint4* sm = (const uint4*)(ring + (size_t)s * kChunkBytes);
        const float2 r = (ALIGNED && nvec == kChunkBytes / 16)
                             ? chunk_stats<ES, GREEDY, kChunkBytes / 16>(sm, nvec, base, -1, 0.f, lane, a.c_hi, a.c_lo)
                             : chunk_stats<ES, GREEDY, 0>(sm, nvec, base, si, sv, lane, a.c_hi, a.c_lo);
        if (lane == 0) partial[(size_t)g * nch + c] = r;
        __syncwarp();
        if (issued < count) issue(s);
        if constexpr (!ALIGNED) __syncwarp();
        advance(cc);
        s = (s + 1 == kStages) ? 0 : s + 1;
    }
    if (failed) {
        // a wait expired: let every copy this warp still has in flight land,
        // the expired one included (each again bounded), so that no copy
        // completes into the shared memory of an exited CTA
        for (int k = 0; k < kStages; ++k)
            if (pending & (1u << k)) mbar_wait_bounded(&bars[k], (phase >> k) & 1u);
        __syncwarp();
    }
    warp_exit(failed);
}

}  // namespace specv
