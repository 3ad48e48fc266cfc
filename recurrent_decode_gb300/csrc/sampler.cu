// sampler.cu -- batched next-token sampling, one CTA (1024 threads) per slot row.
//
// What is sampled follows the Albatross worker loop (RWKV-Runner Albatross
// article, "连续批处理Worker 主循环": presence / frequency penalties, then
// sample_next_tokens_batch with per-slot temperature / top_p / top_k) and the
// adapter's defaults and occurrence decay ("适配器Runner 与异步引擎之间的桥":
// penalty_decay 0.996).  The draw is made exact and order-independent by
// working on integer weights:
//   l_i  = logit_i - ((occ_i > 0 ? presence : 0) + occ_i * frequency)
//   q1_i = floor(2^24 * 2^((l_i - max l) * log2 e))            (fp32 steps, no contraction)
//   top-p keeps q1_i >= tp, tp the largest value whose tail mass reaches
//   ceil(top_p * sum q1), found exactly with a two-level (12 + 12 bit) radix
//   histogram of weight sums; top-k keeps the first k in (q1 desc, index asc)
//   qT_i = floor(2^24 * 2^((l_i - max l) / T * log2 e)) on the kept set
//   r = floor(u * R / 2^64), u one Philox4x32-10 draw (Salmon et al., SC'11),
//   token = first kept index whose running qT sum exceeds r; then
//   occ *= penalty_decay, occ[token] += 1.
// greedy: argmax of the raw logits, lowest index on ties.
#include <cstddef>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/rwkv7.h"
#include "internal.cuh"

namespace rk {

constexpr int SMP_THREADS = 1024;
constexpr int NBUCKET = 4097;  // q1 >> 12 for q1 in [0, 2^24]
// Elements per thread per step of a pass over the row: independent loads issued
// together, so that a pass is not bound by one load's latency at a time.
constexpr int SMP_U = 8;
constexpr int SMP_STEP = SMP_U * SMP_THREADS;

// 2^e for e <= 0: e = n + f (n nearest integer, f exact), 2^f by its degree-7
// Taylor polynomial in f ln 2 (coefficients (ln 2)^k / k!), Horner with fused
// multiply-adds, then an exact scale by 2^n.
__device__ __forceinline__ float exp2_own(float e) {
    if (!(e > -126.0f)) return 0.0f;
    if (e > 0.0f) e = 0.0f;
    const float n = floorf(__fadd_rn(e, 0.5f));
    const float f = __fsub_rn(e, n);
    float z = 0.0000152527338040598403f;
    z = __fmaf_rn(z, f, 0.000154035303933816099f);
    z = __fmaf_rn(z, f, 0.00133335581464284434f);
    z = __fmaf_rn(z, f, 0.00961812910762847717f);
    z = __fmaf_rn(z, f, 0.0555041086648215800f);
    z = __fmaf_rn(z, f, 0.240226506959100712f);
    z = __fmaf_rn(z, f, 0.693147180559945309f);
    z = __fmaf_rn(z, f, 1.0f);
    const float sc = __int_as_float(((int)n + 127) << 23);
    return __fmul_rn(z, sc);
}

__device__ __forceinline__ uint32_t qweight(float l, float m, float T) {
    float dlt = __fsub_rn(l, m);
    if (T != 1.0f) dlt = __fdiv_rn(dlt, T);
    const float e = __fmul_rn(dlt, 1.44269504088896340736f);
    const float pz = exp2_own(e);
    return (uint32_t)floorf(__fmul_rn(pz, 16777216.0f));
}

__device__ __forceinline__ void philox4x32_10(uint32_t c[4], uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t hi0 = __umulhi(0xD2511F53u, c[0]), lo0 = 0xD2511F53u * c[0];
        const uint32_t hi1 = __umulhi(0xCD9E8D57u, c[2]), lo1 = 0xCD9E8D57u * c[2];
        const uint32_t n0 = hi1 ^ c[1] ^ k0, n2 = hi0 ^ c[3] ^ k1;
        c[0] = n0;
        c[1] = lo1;
        c[2] = n2;
        c[3] = lo0;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
}

struct SmpShared {
    // Bucket sums as two 32-bit words (a sum reaches 2^40): native 32-bit
    // shared-memory atomics on the low word, a carry counted in the high word.
    uint32_t hlo[NBUCKET];
    uint32_t hhi[NBUCKET];
    unsigned long long wsum[32];
    float wf[32];
    int wi[32];
    unsigned long long bcast[4];
    int ibcast[4];
};

__device__ __forceinline__ unsigned long long hist_get(const SmpShared &sm, int h) {
    return ((unsigned long long)sm.hhi[h] << 32) | sm.hlo[h];
}
__device__ __forceinline__ void hist_clear(SmpShared &sm) {
    for (int i = threadIdx.x; i < NBUCKET; i += blockDim.x) {
        sm.hlo[i] = 0u;
        sm.hhi[i] = 0u;
    }
}

// Exclusive prefix sum over the CTA (thread order) of a 64-bit value; returns
// the prefix and writes the total to *total.
__device__ __forceinline__ unsigned long long block_excl_scan(unsigned long long v, SmpShared &sm,
                                                              unsigned long long *total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    unsigned long long x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    __syncthreads();
    if (lane == 31) sm.wsum[w] = x;
    __syncthreads();
    if (w == 0) {
        unsigned long long t = sm.wsum[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        sm.wsum[lane] = t;  // inclusive over warps
    }
    __syncthreads();
    const unsigned long long before = (w > 0 ? sm.wsum[w - 1] : 0ull);
    *total = sm.wsum[31];
    return before + x - v;
}

__device__ __forceinline__ unsigned long long block_sum_u64(unsigned long long v, SmpShared &sm) {
    unsigned long long tot;
    block_excl_scan(v, sm, &tot);
    return tot;
}

// Over the 4096 (+1 top) buckets of the histogram: the largest bucket index h with
// base + sum_{h' >= h} hist[h'] >= target (-1 if none); *above receives
// base + sum_{h' > h} hist[h'].  nb = number of buckets (4097 or 4096).
__device__ __forceinline__ int find_cut(SmpShared &sm, int nb, unsigned long long base,
                                        unsigned long long target, unsigned long long *above) {
    // thread t owns buckets [4t, 4t + 4); bucket 4096 (if nb == 4097) is added to base.
    const int t = threadIdx.x;
    unsigned long long top = (nb == NBUCKET) ? hist_get(sm, 4096) : 0ull;
    unsigned long long mine = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) mine += hist_get(sm, 4 * t + j);
    // suffix sum: total - inclusive prefix
    unsigned long long total;
    const unsigned long long excl = block_excl_scan(mine, sm, &total);
    const unsigned long long after_me = total - excl - mine;  // buckets owned by later threads
    if (t == 0) {
        sm.ibcast[0] = -1;
        sm.bcast[0] = 0ull;
    }
    __syncthreads();
    if (nb == NBUCKET && base + top >= target) {
        if (t == 0) {
            sm.ibcast[0] = 4096;
            sm.bcast[0] = base;
        }
    } else {
        unsigned long long run = base + top + after_me;
        for (int j = 3; j >= 0; --j) {
            const int h = 4 * t + j;
            const unsigned long long above_h = run;
            run += hist_get(sm, h);
            if (run >= target && above_h < target) {
                sm.ibcast[0] = h;  // unique: the suffix sum crosses target exactly once
                sm.bcast[0] = above_h;
            }
        }
    }
    __syncthreads();
    *above = sm.bcast[0];
    const int h = sm.ibcast[0];
    __syncthreads();
    return h;
}

// hist[key] += val for the lanes with live set.  The weights of a row crowd
// into few low buckets when the logits are spread wide, and per-lane atomics on
// one address serialise, so the lanes that share lane 0's key are summed first
// (__reduce_add_sync; val <= 2^24, so 32 of them fit in 32 bits) and added
// once; the others add their own value (distinct keys hit distinct words).
// Sums use native 32-bit shared-memory atomics on the low word, a wrap of it
// is carried into the high word.  Called by all 32 lanes.
__device__ __forceinline__ void hist_add(SmpShared &sm, uint32_t key, uint32_t val) {
    const uint32_t old = atomicAdd(&sm.hlo[key], val);
    if (old + val < old) atomicAdd(&sm.hhi[key], 1u);  // the low word wrapped
}
__device__ __forceinline__ void hist_add_warp(SmpShared &sm, uint32_t key, uint32_t val, bool live) {
    const uint32_t k = live ? key : 0xffffffffu;
    const uint32_t k0 = __shfl_sync(0xffffffffu, k, 0);
    const bool same = k == k0;
    const uint32_t gsum = __reduce_add_sync(0xffffffffu, same ? val : 0u);
    if ((threadIdx.x & 31) == 0) {
        if (live) hist_add(sm, key, gsum);
    } else if (!same && live) {
        hist_add(sm, key, val);
    }
}

// MINB CTAs per SM.  Batches with more rows than SMs take the two-CTA build
// (32 registers a thread, a few spilled), so that up to two rows per SM run as
// one wave -- at B=256 165 us against 185 us for two waves; smaller batches
// keep the one-CTA build (64 registers), whose greedy path is ~3 us faster.
template <int MINB>
__global__ void __launch_bounds__(SMP_THREADS, MINB) sampler_kernel(const SamplerParams p) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    SmpShared &sm = *reinterpret_cast<SmpShared *>(smem_raw);
    const int b = blockIdx.x, tid = threadIdx.x;
    if (tid == 0) tl_start(p.tl);
    pdl_wait();
    pdl_launch();
    if (tid == 0) tl_release(p.tl);
    const int slot = p.slots[b];
    if (slot < 0 || slot >= p.n_slots) {
        if (tid == 0) {
            atomicOr(p.err, ERR_SLOT);
            p.next[b] = 0;
        }
        return;
    }
    const SampleParamsDev sp = p.params[slot];
    const int V = p.V;
    const float *lg = p.logits + (size_t)b * V;

    if (sp.greedy || !(sp.temperature > 0.0f)) {
        float best = -INFINITY;
        int bi = 0x7fffffff;
        for (int i0 = 0; i0 < V; i0 += SMP_STEP) {
            float v[SMP_U];
#pragma unroll
            for (int u = 0; u < SMP_U; ++u) {
                const int i = i0 + u * SMP_THREADS + tid;
                v[u] = i < V ? lg[i] : -INFINITY;
            }
#pragma unroll
            for (int u = 0; u < SMP_U; ++u) {  // ascending i per thread: ">" keeps the lowest index
                const int i = i0 + u * SMP_THREADS + tid;
                if (i < V && (v[u] > best || (v[u] == best && i < bi))) {
                    best = v[u];
                    bi = i;
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, best, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > best || (ov == best && oi < bi)) {
                best = ov;
                bi = oi;
            }
        }
        if ((tid & 31) == 0) {
            sm.wf[tid >> 5] = best;
            sm.wi[tid >> 5] = bi;
        }
        __syncthreads();
        if (tid == 0) {
            float bv = sm.wf[0];
            int bj = sm.wi[0];
            for (int w = 1; w < 32; ++w)
                if (sm.wf[w] > bv || (sm.wf[w] == bv && sm.wi[w] < bj)) {
                    bv = sm.wf[w];
                    bj = sm.wi[w];
                }
            p.next[b] = (bj < V) ? bj : 0;
            tl_end(p.tl);
        }
        return;
    }

    float *occ = p.occ + (size_t)slot * V;
    float *lp = p.lpen + (size_t)b * V;
    // ---- pass A: penalty and max; the occurrence counts are decayed here
    // (every row draws a token: the row maximum always keeps weight 2^24), the
    // drawn token's +1 is added at the end.
    float mx = -INFINITY;
    for (int i0 = 0; i0 < V; i0 += SMP_STEP) {
        float lv[SMP_U], ov[SMP_U];
#pragma unroll
        for (int u = 0; u < SMP_U; ++u) {
            const int i = i0 + u * SMP_THREADS + tid;
            lv[u] = i < V ? lg[i] : 0.0f;
            ov[u] = i < V ? occ[i] : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < SMP_U; ++u) {
            const int i = i0 + u * SMP_THREADS + tid;
            if (i < V) {
                const float pres = ov[u] > 0.0f ? sp.presence : 0.0f;
                float t = __fmul_rn(ov[u], sp.frequency);
                t = __fadd_rn(pres, t);
                const float l = __fsub_rn(lv[u], t);
                lp[i] = l;
                mx = fmaxf(mx, l);
                occ[i] = __fmul_rn(ov[u], sp.penalty_decay);
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if ((tid & 31) == 0) sm.wf[tid >> 5] = mx;
    __syncthreads();
    if (tid == 0) {
        float m = sm.wf[0];
        for (int w = 1; w < 32; ++w) m = fmaxf(m, sm.wf[w]);
        sm.wf[0] = m;
    }
    __syncthreads();
    const float m = sm.wf[0];
    __syncthreads();

    // ---- pass B: weight sums per (q1 >> 12) bucket
    hist_clear(sm);
    __syncthreads();
    // At temperature 1 the draw weights are the q1 weights, so they are
    // computed once here and stored over the row's penalised logits; the later
    // passes read them back.  Otherwise every pass recomputes them from lp.
    const bool t1 = sp.temperature == 1.0f;
    uint32_t *lq = reinterpret_cast<uint32_t *>(lp);
    unsigned long long q1loc = 0;
    for (int i0 = 0; i0 < V; i0 += SMP_STEP) {  // warp-uniform trip count
        float lv[SMP_U];
#pragma unroll
        for (int u = 0; u < SMP_U; ++u) {
            const int i = i0 + u * SMP_THREADS + tid;
            lv[u] = i < V ? lp[i] : -INFINITY;
        }
#pragma unroll
        for (int u = 0; u < SMP_U; ++u) {
            const int i = i0 + u * SMP_THREADS + tid;
            uint32_t q = 0;
            if (i < V) {
                q = qweight(lv[u], m, 1.0f);
                if (t1) lq[i] = q;
                q1loc += q;
            }
            hist_add_warp(sm, q >> 12, q, q != 0u);
        }
    }
    const unsigned long long Q1 = block_sum_u64(q1loc, sm);
    unsigned long long target = (unsigned long long)ceil(__dmul_rn((double)sp.top_p, (double)Q1));
    if (target < 1ull) target = 1ull;
    if (target > Q1) target = Q1;
    unsigned long long above;
    const int hb = find_cut(sm, NBUCKET, 0ull, target, &above);
    // q1 of element i, read back (temperature 1) or recomputed
    auto q1_at = [&](int i) -> uint32_t { return t1 ? lq[i] : qweight(lp[i], m, 1.0f); };
    // ---- pass C: low 12 bits within bucket hb
    hist_clear(sm);
    __syncthreads();
    for (int i0 = 0; i0 < V; i0 += SMP_STEP) {
        uint32_t qv[SMP_U];
#pragma unroll
        for (int u = 0; u < SMP_U; ++u) {
            const int i = i0 + u * SMP_THREADS + tid;
            qv[u] = i < V ? q1_at(i) : 0u;
        }
#pragma unroll
        for (int u = 0; u < SMP_U; ++u)
            hist_add_warp(sm, qv[u] & 4095u, qv[u], (int)(qv[u] >> 12) == hb && qv[u] != 0u);
    }
    __syncthreads();
    unsigned long long above2;
    const int lo = find_cut(sm, 4096, above, target, &above2);
    const uint32_t tp = ((uint32_t)hb << 12) | (uint32_t)(lo < 0 ? 0 : lo);

    // ---- optional top-k: t_k = k-th largest q1 (counts), ties by lowest index
    const bool use_k = sp.top_k > 0 && sp.top_k < V;
    uint32_t tk = 0;
    unsigned long long need_ties = 0;
    if (use_k) {
        const unsigned long long K = (unsigned long long)sp.top_k;
        hist_clear(sm);
        __syncthreads();
        for (int i0 = 0; i0 < V; i0 += SMP_STEP) {
            uint32_t qv[SMP_U];
#pragma unroll
            for (int u = 0; u < SMP_U; ++u) {
                const int i = i0 + u * SMP_THREADS + tid;
                qv[u] = i < V ? q1_at(i) : 0u;
            }
#pragma unroll
            for (int u = 0; u < SMP_U; ++u) hist_add_warp(sm, qv[u] >> 12, 1u, i0 + u * SMP_THREADS + tid < V);
        }
        __syncthreads();
        unsigned long long cabove;
        const int hk = find_cut(sm, NBUCKET, 0ull, K, &cabove);
        hist_clear(sm);
        __syncthreads();
        for (int i0 = 0; i0 < V; i0 += SMP_STEP) {
            uint32_t qv[SMP_U];
#pragma unroll
            for (int u = 0; u < SMP_U; ++u) {
                const int i = i0 + u * SMP_THREADS + tid;
                qv[u] = i < V ? q1_at(i) : 0u;
            }
#pragma unroll
            for (int u = 0; u < SMP_U; ++u)
                hist_add_warp(sm, qv[u] & 4095u, 1u,
                              i0 + u * SMP_THREADS + tid < V && (int)(qv[u] >> 12) == hk);
        }
        __syncthreads();
        unsigned long long cgt;
        const int lk = find_cut(sm, 4096, cabove, K, &cgt);
        tk = ((uint32_t)hk << 12) | (uint32_t)(lk < 0 ? 0 : lk);
        need_ties = K - cgt;  // elements equal to tk to keep (lowest indices first)
    }

    // ---- pass D: kept set, qT, exclusive scan in index order, draw, pick.
    // Warp w owns the contiguous range [w * CW, (w + 1) * CW) and walks it in
    // blocks of 32 consecutive elements (one coalesced load per block), so the
    // index order is (warp, block, lane).  A tie with t_k is kept while fewer
    // than need_ties ties precede it in that order.
    const int lane = tid & 31, w = tid >> 5;
    const unsigned lt_mask = (1u << lane) - 1u;
    const int CW = ((V + 31) / 32 + 31) / 32 * 32;
    const int w_lo = w * CW, w_hi = min(V, w_lo + CW);
    const int nblk = w_hi > w_lo ? (w_hi - w_lo + 31) / 32 : 0;  // warp-uniform
    unsigned long long tie_base = 0;  // ties before this warp's range
    if (use_k) {
        unsigned ties = 0;
        for (int k0 = 0; k0 < nblk; k0 += SMP_U) {
            uint32_t qv[SMP_U];
#pragma unroll
            for (int u = 0; u < SMP_U; ++u) {
                const int i = w_lo + (k0 + u) * 32 + lane;
                qv[u] = (k0 + u < nblk && i < w_hi) ? q1_at(i) : 0u;
            }
#pragma unroll
            for (int u = 0; u < SMP_U; ++u) {
                const int i = w_lo + (k0 + u) * 32 + lane;
                ties += (k0 + u < nblk && i < w_hi && qv[u] == tk) ? 1u : 0u;
            }
        }
        const unsigned wt = __reduce_add_sync(0xffffffffu, ties);
        unsigned long long tt;
        tie_base = __shfl_sync(0xffffffffu, block_excl_scan(lane == 0 ? (unsigned long long)wt : 0ull, sm, &tt), 0);
    }
    // kept weight of element i with value q; *tie_seen counts the warp's ties so far
    auto kept_weight = [&](int i, bool in, uint32_t q, unsigned long long *tie_seen) -> unsigned long long {
        bool keep = in && q >= tp;
        if (use_k) {
            const bool tie = in && q == tk;
            const unsigned tb = __ballot_sync(0xffffffffu, tie);
            const unsigned long long rank = *tie_seen + (unsigned long long)__popc(tb & lt_mask);
            keep = keep && (q > tk || (tie && rank < need_ties));
            *tie_seen += (unsigned long long)__popc(tb);
        }
        if (!keep) return 0ull;
        return t1 ? (unsigned long long)q : (unsigned long long)qweight(lp[i], m, sp.temperature);
    };
    unsigned long long rloc = 0;
    {
        unsigned long long tie_seen = tie_base;
        for (int k0 = 0; k0 < nblk; k0 += SMP_U) {
            uint32_t qv[SMP_U];
#pragma unroll
            for (int u = 0; u < SMP_U; ++u) {
                const int i = w_lo + (k0 + u) * 32 + lane;
                qv[u] = (k0 + u < nblk && i < w_hi) ? q1_at(i) : 0u;
            }
#pragma unroll
            for (int u = 0; u < SMP_U; ++u) {
                const int i = w_lo + (k0 + u) * 32 + lane;
                if (k0 + u < nblk) rloc += kept_weight(i, i < w_hi, qv[u], &tie_seen);
            }
        }
    }
    unsigned long long wsum = rloc;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
    unsigned long long R;
    const unsigned long long rbase =
        __shfl_sync(0xffffffffu, block_excl_scan(lane == 0 ? wsum : 0ull, sm, &R), 0);  // before this warp
    const unsigned long long nd = p.ndraw[slot];
    uint32_t ctr[4] = {(uint32_t)nd, (uint32_t)(nd >> 32), 0u, 0u};
    philox4x32_10(ctr, (uint32_t)sp.seed, (uint32_t)(sp.seed >> 32));
    const unsigned long long u64 = (unsigned long long)ctr[0] | ((unsigned long long)ctr[1] << 32);
    const unsigned long long r = __umul64hi(u64, R);
    if (tid == 0) sm.ibcast[1] = -1;
    __syncthreads();
    if (wsum > 0 && rbase <= r && r < rbase + wsum) {  // warp-uniform: this warp holds the draw
        unsigned long long acc = rbase, tie_seen = tie_base;
        bool found = false;
        for (int k0 = 0; k0 < nblk && !found; k0 += SMP_U) {
            uint32_t qv[SMP_U];
#pragma unroll
            for (int u = 0; u < SMP_U; ++u) {
                const int i = w_lo + (k0 + u) * 32 + lane;
                qv[u] = (k0 + u < nblk && i < w_hi) ? q1_at(i) : 0u;
            }
#pragma unroll
            for (int u = 0; u < SMP_U; ++u) {
                if (found || k0 + u >= nblk) continue;  // warp-uniform conditions
                const int i = w_lo + (k0 + u) * 32 + lane;
                const unsigned long long kw = kept_weight(i, i < w_hi, qv[u], &tie_seen);
                unsigned long long incl = kw;  // inclusive scan over the block's lanes
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += y;
                }
                const unsigned hit = __ballot_sync(0xffffffffu, kw > 0 && acc + incl > r);
                if (hit) {
                    if (lane == __ffs(hit) - 1) sm.ibcast[1] = i;
                    found = true;
                }
                acc += __shfl_sync(0xffffffffu, incl, 31);
            }
        }
    }
    __syncthreads();
    const int tok = sm.ibcast[1];
    // ---- pass E: count the drawn token (the decay was applied in pass A)
    if (tid == 0) {
        if (tok >= 0) occ[tok] = __fadd_rn(occ[tok], 1.0f);
        p.next[b] = tok >= 0 ? tok : 0;
        if (tok < 0) atomicOr(p.err, ERR_CONFIG);
        p.ndraw[slot] = nd + 1ull;
        tl_end(p.tl);
    }
}

void launch_sampler(const SamplerParams &p, const LaunchCfg &lc, cudaError_t *e) {
    const size_t smem = sizeof(SmpShared);
    int dev = 0, nsm = 0;
    cudaError_t r0 = cudaGetDevice(&dev);
    if (r0 == cudaSuccess) r0 = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (r0 != cudaSuccess) {
        *e = r0;
        return;
    }
    const bool two = p.B > nsm;
    const void *kfn = two ? (const void *)sampler_kernel<2> : (const void *)sampler_kernel<1>;
    {
        cudaError_t r = ensure_smem_attr(kfn, (int)smem);
        if (r != cudaSuccess) {
            *e = r;
            return;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.B);
    cfg.blockDim = dim3(SMP_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = lc.stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = lc.pdl ? 1 : 0;
    cudaError_t r = two ? cudaLaunchKernelEx(&cfg, sampler_kernel<2>, p) : cudaLaunchKernelEx(&cfg, sampler_kernel<1>, p);
    if (r != cudaSuccess) *e = r;
}

}  // namespace rk

// ---------------------------------------------------------------------------
// rwkv7_sample_rows_static: the sampler above for callers that must not
// allocate device memory (a process whose HBM already belongs to its own
// arena, or a serving loop that cannot take the device-wide synchronisation
// cudaMalloc / cudaFree may cause).  The penalised-logit scratch the kernel
// needs ([B][V] fp32) comes from this fixed module array instead of a ctx
// buffer; the CUDA runtime reserves it on each device that loads the library
// and keeps it until the process exits.  The kernel and its arithmetic are the
// ones rwkv7_sample_batch launches.
namespace {

constexpr size_t STATIC_LPEN_ELEMS = (size_t)RWKV7_SAMPLE_STATIC_MAX_ELEMS;  // 16 MiB of fp32
constexpr int STATIC_MAX_DEVICES = 64;

// The scratch array.  In host code this name is only a stand-in for the device
// symbol: its device address comes from cudaGetSymbolAddress, per device.
static __device__ __align__(256) float g_static_lpen[STATIC_LPEN_ELEMS];

std::mutex g_static_mu;
float *g_static_lpen_dev[STATIC_MAX_DEVICES] = {};  // device address of g_static_lpen, per device
thread_local char g_static_msg[192];

// The public parameter struct is handed to the kernel as its device copy.
static_assert(sizeof(rwkv7_sampling) == sizeof(rk::SampleParamsDev), "sampling struct size");
static_assert(offsetof(rwkv7_sampling, top_k) == offsetof(rk::SampleParamsDev, top_k), "top_k offset");
static_assert(offsetof(rwkv7_sampling, penalty_decay) == offsetof(rk::SampleParamsDev, penalty_decay),
              "penalty_decay offset");
static_assert(offsetof(rwkv7_sampling, seed) == offsetof(rk::SampleParamsDev, seed), "seed offset");
static_assert(offsetof(rwkv7_sampling, greedy) == offsetof(rk::SampleParamsDev, greedy), "greedy offset");

int static_fail(const char **err_msg, int code, const char *fmt, long long a = 0, long long b = 0) {
    snprintf(g_static_msg, sizeof g_static_msg, fmt, a, b);
    if (err_msg) *err_msg = g_static_msg;
    return code;
}

// Once per device, with that device current: look up the scratch's device
// address and allow the kernel its dynamic shared memory on this device.
int static_setup(float **lpen, const char **err_msg) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return static_fail(err_msg, RWKV7_ECUDA, "cudaGetDevice failed (error %lld)", (long long)e);
    if (dev < 0 || dev >= STATIC_MAX_DEVICES)
        return static_fail(err_msg, RWKV7_EINVAL, "device ordinal %lld beyond the supported %lld", dev,
                           STATIC_MAX_DEVICES);
    std::lock_guard<std::mutex> lk(g_static_mu);
    if (!g_static_lpen_dev[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_lpen);
        if (e != cudaSuccess || !p)
            return static_fail(err_msg, RWKV7_ECUDA, "cudaGetSymbolAddress of the sampler scratch failed (error %lld)",
                               (long long)e);
        e = cudaFuncSetAttribute(rk::sampler_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)sizeof(rk::SmpShared));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(rk::sampler_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)sizeof(rk::SmpShared));
        if (e != cudaSuccess)
            return static_fail(err_msg, RWKV7_ECUDA, "setting the sampler's shared-memory limit failed (error %lld)",
                               (long long)e);
        g_static_lpen_dev[dev] = static_cast<float *>(p);
    }
    *lpen = g_static_lpen_dev[dev];
    return RWKV7_OK;
}

}  // namespace

extern "C" int rwkv7_sample_rows_static(const float *d_logits, const int32_t *d_rows, int32_t B, int32_t V,
                                        int32_t n_rows, float *d_occ, const rwkv7_sampling *d_params,
                                        uint64_t *d_ndraw, int32_t *d_next_out, uint32_t *d_err,
                                        void *cuda_stream, const char **err_msg) {
    if (err_msg) *err_msg = "";
    if (!d_logits || !d_rows || !d_occ || !d_params || !d_ndraw || !d_next_out || !d_err)
        return static_fail(err_msg, RWKV7_EINVAL, "null pointer argument");
    if (((uintptr_t)d_params & 7u) || ((uintptr_t)d_ndraw & 7u))
        return static_fail(err_msg, RWKV7_EINVAL, "d_params and d_ndraw must be 8-byte aligned");
    if (B < 1 || V < 1 || n_rows < 1)
        return static_fail(err_msg, RWKV7_EINVAL, "B, V and n_rows must be >= 1 (B=%lld, V=%lld)", B, V);
    if ((size_t)B * (size_t)V > STATIC_LPEN_ELEMS)
        return static_fail(err_msg, RWKV7_EINVAL,
                           "B * V = %lld exceeds the static sampler scratch of %lld fp32 elements; split the batch",
                           (long long)B * V, (long long)STATIC_LPEN_ELEMS);
    float *lpen = nullptr;
    int rc = static_setup(&lpen, err_msg);
    if (rc) return rc;
    rk::SamplerParams sp;
    memset(&sp, 0, sizeof sp);
    sp.B = B;
    sp.V = V;
    sp.n_slots = n_rows;
    sp.slots = d_rows;
    sp.logits = d_logits;
    sp.occ = d_occ;
    sp.params = reinterpret_cast<const rk::SampleParamsDev *>(d_params);
    sp.ndraw = reinterpret_cast<unsigned long long *>(d_ndraw);
    sp.lpen = lpen;  // rows b use [b*V, (b+1)*V), inside the array since B*V <= its size
    sp.next = d_next_out;
    sp.err = d_err;
    cudaError_t e = cudaSuccess;
    rk::launch_sampler(sp, rk::LaunchCfg{static_cast<cudaStream_t>(cuda_stream), false}, &e);
    if (e != cudaSuccess)
        return static_fail(err_msg, RWKV7_ECUDA, "sampler launch failed (error %lld)", (long long)e);
    return RWKV7_OK;
}
