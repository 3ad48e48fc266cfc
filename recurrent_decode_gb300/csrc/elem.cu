// elem.cu -- per-slot kernels of the decode step that are not matrix products:
// embedding + LayerNorm, LayerNorm + token-shift mixes, the WKV7 state update
// with GroupNorm / bonus / output gate, and slot-pool maintenance.
//
// The pages fuse LayerNorm with the token-shift mixes for T=1 decode
// ("RWKV 批量推理中 Prefill 的正确打开方式", §三: fused_ln_tmix_mix / LN1_TMIX_FUSE
// for the time mix, add_layer_norm_cmix_mix_f16 for the channel mix); the
// same fusion is kept here, one CTA per slot row.
#include "internal.cuh"

namespace rk {

// LayerNorm kernels: one CTA per slot row, 8 consecutive elements per thread
// (16-byte loads), blockDim = d/8 rounded up to a warp.
__device__ __forceinline__ void h8_to_f(const uint4 &u, float (&f)[8]) {
    const __half2 *h = reinterpret_cast<const __half2 *>(&u);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 t = __half22float2(h[k]);
        f[2 * k] = t.x;
        f[2 * k + 1] = t.y;
    }
}
__device__ __forceinline__ uint4 f_to_h8(const float (&f)[8]) {
    uint4 u;
    __half2 *h = reinterpret_cast<__half2 *>(&u);
#pragma unroll
    for (int k = 0; k < 4; ++k) h[k] = __floats2half2_rn(f[2 * k], f[2 * k + 1]);
    return u;
}
__device__ __forceinline__ void ld8f(const float *p, float (&f)[8]) {
    const float4 a = *reinterpret_cast<const float4 *>(p), b = *reinterpret_cast<const float4 *>(p + 4);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}
__device__ __forceinline__ void st8f(float *p, const float (&f)[8]) {
    *reinterpret_cast<float4 *>(p) = make_float4(f[0], f[1], f[2], f[3]);
    *reinterpret_cast<float4 *>(p + 4) = make_float4(f[4], f[5], f[6], f[7]);
}

// x[8] += sum over j < nsplit of part[j * stride + off .. +8], slabs added in
// order j = 0, 1, ... (the loads of up to eight slabs are issued together).
__device__ __forceinline__ void add_slabs(float (&x)[8], const float *part, int nsplit, long long stride, size_t off) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    int j = 0;
    for (; j + 8 <= nsplit; j += 8) {
        float t[8][8];
#pragma unroll
        for (int u = 0; u < 8; ++u) ld8f(part + (size_t)(j + u) * stride + off, t[u]);
#pragma unroll
        for (int u = 0; u < 8; ++u)
#pragma unroll
            for (int k = 0; k < 8; ++k) acc[k] += t[u][k];
    }
    if (j + 4 <= nsplit) {
        float t[4][8];
#pragma unroll
        for (int u = 0; u < 4; ++u) ld8f(part + (size_t)(j + u) * stride + off, t[u]);
        float t2[3][8];
        const int rest = nsplit - j - 4;  // 0..3 more slabs, loaded alongside
#pragma unroll
        for (int u = 0; u < 3; ++u)
            if (u < rest) ld8f(part + (size_t)(j + 4 + u) * stride + off, t2[u]);
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int k = 0; k < 8; ++k) acc[k] += t[u][k];
#pragma unroll
        for (int u = 0; u < 3; ++u)
            if (u < rest)
#pragma unroll
                for (int k = 0; k < 8; ++k) acc[k] += t2[u][k];
        j = nsplit;
    }
    for (; j < nsplit; ++j) {
        float t[8];
        ld8f(part + (size_t)j * stride + off, t);
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[k] += t[k];
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) x[k] += acc[k];
}

// Count, sum and sum of squared deviations of a set of values (Chan, Golub and
// LeVeque's pairwise update), for the WKV kernel's GroupNorm.  The merge is
// symmetric in its operands -- (sa nb - sb na)^2 is the same number either way
// round -- so every lane of a butterfly ends with the same bits.
struct Moments {
    float n, s, m2;
};
__device__ __forceinline__ Moments merge_moments(const Moments &a, const Moments &b) {
    Moments r;
    r.n = a.n + b.n;
    r.s = a.s + b.s;
    r.m2 = a.m2 + b.m2;
    if (a.n > 0.0f && b.n > 0.0f) {
        const float t = a.s * b.n - b.s * a.n;
        r.m2 += t * t / (a.n * b.n * r.n);
    }
    return r;
}

// Sum over the CTA with one barrier.  `red` holds 32 floats.  A thread may
// write them while others still read the previous sum from the same buffer,
// so consecutive sums alternate between two buffers: a thread writes buffer A
// again only after the barrier of the sum on buffer B, which every thread
// reaches after reading A.
__device__ __forceinline__ float block_sum(float v, float *red) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    v = warp_sum(v);
    if (lane == 0) red[w] = v;
    __syncthreads();
    float t = 0.0f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) t += red[i];
    return t;
}

// In-place LayerNorm of the d values held 8 per thread (inactive threads hold
// zeros): (x - mean) / sqrt(var + 1e-5) * w + b, biased variance.  `red` holds
// 64 floats.  Two barriers (mean, then the centred sum of squares): a
// single-barrier form merging (count, sum, squared deviations) pairwise
// measured slower (2.9B 4.2 us a launch against 3.6).
__device__ __forceinline__ void ln8(float (&v)[8], bool act, int d, const uint4 &w4, const uint4 &b4, float *red) {
    float s = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) s += v[k];
    const float mean = block_sum(s, red) / (float)d;
    float q = 0.0f;
    if (act) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float t = v[k] - mean;
            q += t * t;
        }
    }
    const float var = block_sum(q, red + 32) / (float)d;
    const float rs = 1.0f / sqrtf(var + 1e-5f);
    float w[8], b[8];
    h8_to_f(w4, w);
    h8_to_f(b4, b);
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] = (v[k] - mean) * rs * w[k] + b[k];
}

// x[b] = LN0(emb[token[b]]).  Also validates the step's slots and tokens:
// range errors are latched and the row falls back to token 0; CTA 0 looks for
// repeated slots with a bitmap in shared memory.
__global__ void embed_kernel(const ElemParams p) {
    extern __shared__ uint32_t bitmap[];
    __shared__ float red[64];
    if (threadIdx.x == 0) tl_start(p.tl);
    pdl_wait();
    pdl_launch();
    if (threadIdx.x == 0) tl_release(p.tl);
    const int b = blockIdx.x;
    const int i0 = threadIdx.x * 8;
    const bool act = i0 < p.d;
    const int slot = p.single_slot >= 0 ? p.single_slot : p.slots[b];
    int tok = p.tokens[b];
    if (threadIdx.x == 0) {
        if (slot < 0 || slot >= p.n_slots) atomicOr(p.err, ERR_SLOT);
        if (tok < 0 || tok >= p.V) atomicOr(p.err, ERR_TOKEN);
    }
    if (tok < 0 || tok >= p.V) tok = 0;
    float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    uint4 w4 = make_uint4(0, 0, 0, 0), b4 = w4;
    if (act) {
        h8_to_f(*reinterpret_cast<const uint4 *>(p.emb + (size_t)tok * p.d + i0), v);
        w4 = *reinterpret_cast<const uint4 *>(p.ln_w + i0);
        b4 = *reinterpret_cast<const uint4 *>(p.ln_b + i0);
    }
    ln8(v, act, p.d, w4, b4, red);
    if (act) st8f(p.x + (size_t)b * p.d + i0, v);
    if (threadIdx.x == 0) tl_end(p.tl);
    if (b == 0 && p.single_slot < 0) {
        const int words = (p.n_slots + 31) / 32;
        for (int i = threadIdx.x; i < words; i += blockDim.x) bitmap[i] = 0u;
        __syncthreads();
        for (int i = threadIdx.x; i < p.B; i += blockDim.x) {
            const int s = p.slots[i];
            if (s >= 0 && s < p.n_slots) {
                const uint32_t bit = 1u << (s & 31);
                if (atomicOr(&bitmap[s >> 5], bit) & bit) atomicOr(p.err, ERR_DUP);
            }
        }
    }
}

// xl = LN(x[b]); for each mix q: xo[q][b] = fp16(xl + (shift - xl) * mu_q); shift <- xl.
// NMIX = 6 for the time mix (r, w, k, v, a, g), 1 for the channel mix.  The
// constants and the shift state (written only by this kernel, one step
// earlier) are fetched before the dependency wait.  Rows of up to 512 threads
// (d <= 4096); bounded at that size the compiler takes up to 128 registers and
// keeps more loads in flight (2.9B: 3.55 us a launch against 4.40 unbounded).
// A two-rows-per-SM build for wide batches (64 registers, spills) measured
// slower at 7.2B, B=256 (10.2 us against 8.8).
template <int NMIX>
__global__ void __launch_bounds__(512, 1) ln_mix_kernel(const ElemParams p) {
    __shared__ float red[64];
    if (threadIdx.x == 0) tl_start(p.tl);
    const int b = blockIdx.x;
    const int i0 = threadIdx.x * 8;
    const bool act = i0 < p.d;
    const int slot = p.slots[b];
    const bool ok = slot >= 0 && slot < p.n_slots;
    uint4 w4 = make_uint4(0, 0, 0, 0), b4 = w4, mu4[NMIX];
    float sh[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float *shp = p.shift + (size_t)(ok ? slot : 0) * p.d + i0;
    if (act) {
        w4 = *reinterpret_cast<const uint4 *>(p.ln_w + i0);
        b4 = *reinterpret_cast<const uint4 *>(p.ln_b + i0);
#pragma unroll
        for (int q = 0; q < NMIX; ++q) mu4[q] = *reinterpret_cast<const uint4 *>(p.mu[q] + i0);
        if (ok) ld8f(shp, sh);
    }
    // Dependents may launch as soon as every row has started: the GEMM that
    // follows then fetches its first weight stages while this kernel waits.
    pdl_launch();
    pdl_wait();
    if (threadIdx.x == 0) tl_release(p.tl);
    float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (act) {
        ld8f(p.x + (size_t)b * p.d + i0, v);
        if (p.part) {
            add_slabs(v, p.part, p.nsplit, p.split_stride, (size_t)b * p.d + i0);
            st8f(p.x + (size_t)b * p.d + i0, v);
        }
    }
    ln8(v, act, p.d, w4, b4, red);
    if (!act) return;
#pragma unroll
    for (int q = 0; q < NMIX; ++q) {
        float mu[8], o[8];
        h8_to_f(mu4[q], mu);
#pragma unroll
        for (int k = 0; k < 8; ++k) o[k] = v[k] + (sh[k] - v[k]) * mu[k];
        *reinterpret_cast<uint4 *>(p.xo[q] + (size_t)b * p.d + i0) = f_to_h8(o);
    }
    if (ok) st8f(shp, v);
    if (threadIdx.x == 0) tl_end(p.tl);
}

// xo[0][b] = fp16(LN_out(x[b])): the input of the head projection.
__global__ void ln_out_kernel(const ElemParams p) {
    __shared__ float red[64];
    if (threadIdx.x == 0) tl_start(p.tl);
    const int b = blockIdx.x;
    const int i0 = threadIdx.x * 8;
    const bool act = i0 < p.d;
    uint4 w4 = make_uint4(0, 0, 0, 0), b4 = w4;
    if (act) {
        w4 = *reinterpret_cast<const uint4 *>(p.ln_w + i0);
        b4 = *reinterpret_cast<const uint4 *>(p.ln_b + i0);
    }
    pdl_launch();  // the head GEMM may launch and prefetch while this waits
    pdl_wait();
    if (threadIdx.x == 0) tl_release(p.tl);
    float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (act) {
        ld8f(p.x + (size_t)b * p.d + i0, v);
        if (p.part) add_slabs(v, p.part, p.nsplit, p.split_stride, (size_t)b * p.d + i0);
    }
    ln8(v, act, p.d, w4, b4, red);
    if (act) *reinterpret_cast<uint4 *>(p.xo[0] + (size_t)b * p.d + i0) = f_to_h8(v);
    if (threadIdx.x == 0) tl_end(p.tl);
}

static int ln_threads(int d) { return ((d / 8) + 31) / 32 * 32; }

// ---------------------------------------------------------------------------
// WKV7: one CTA per (head h, slot row b), 128 threads.  The pair's 16 KB fp32
// state lands in shared memory through one bulk copy issued before the
// dependency wait (only this kernel, one step earlier, writes it), so registers
// stay few and up to 12 CTAs -- 192 KB of state reads -- are in flight per SM.
//   kh = normalize(k * k_k), kp = k * (1 + (a - 1) * k_a),
//   vp = v (layer 0, also stored as v_first) or v + (v_first - v) * vg,
//   S[i][j] <- S[i][j] dec_j - (sum_m S[i][m] kh_m) kh_j a_j + vp_i kp_j,
//   y_i = sum_j S[i][j] r_j,
//   z = (GroupNorm(y) * gamma + beta + (sum_j r_j kp_j r_k_j) vp) * g  -> fp16.
// Thread t updates rows t/16 + 8q (q < 8) at columns 4(t % 16)..+3: the 16
// lanes of a half-warp own a whole row (row reductions are 4 shuffles) and
// write it back as one contiguous 256-byte segment with streaming stores.
// ---------------------------------------------------------------------------
constexpr int WKV_THREADS = 128;
struct WkvSmem {
    float st[HS * HS];
    alignas(16) float kh[HS];
    alignas(16) float ka[HS];
    alignas(16) float dec[HS];
    alignas(16) float kp[HS];
    alignas(16) float vp[HS];
    alignas(16) float r[HS];
    alignas(16) float y[HS];
    float red[8];
    uint64_t full;
    uint32_t ok;
};

__device__ __forceinline__ float sum64(float v, float *s2, int barid) {
    v = warp_sum(v);
    if ((threadIdx.x & 31) == 0) s2[threadIdx.x >> 5] = v;
    named_bar(barid, 64);
    const float t = s2[0] + s2[1];
    named_bar(barid, 64);
    return t;
}

__global__ void __launch_bounds__(WKV_THREADS, 12) wkv_kernel(const WkvParams p) {
    extern __shared__ __align__(128) uint8_t wkv_raw[];
    WkvSmem &sm = *reinterpret_cast<WkvSmem *>(wkv_raw);
    const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
    const int slot = p.slots[b];
    const bool ok = slot >= 0 && slot < p.n_slots;
    float *S = p.wkv + ((size_t)(ok ? slot : 0) * p.H + h) * (HS * HS);
    if (tid == 0) {
        tl_start(p.tl);
        sm.ok = 0u;
        mbar_init(&sm.full, 1);
        fence_barrier_init();
        mbar_expect_tx(&sm.full, HS * HS * 4);
        bulk_g2s(sm.st, S, HS * HS * 4, &sm.full);
    }
    // the layer's per-channel constants, before the dependency wait (kept as
    // fp16 pairs: the registers live across the state update)
    const int c = h * HS + (tid & (HS - 1));
    __half2 kkka = __float2half2_rn(0.f), rkg = kkka, lnwb = kkka;
    if (tid < HS) {
        kkka = __halves2half2(p.k_k[c], p.k_a[c]);
        rkg = __halves2half2(p.r_k[c], p.r_k[c]);
        lnwb = __halves2half2(p.lnx_w[c], p.lnx_b[c]);
    }
    pdl_wait();
    pdl_launch();
    if (tid == 0) tl_release(p.tl);

    const size_t off = (size_t)b * p.d + (size_t)h * HS;
    float rv = 0.f, kpv = 0.f, vpv = 0.f;
    if (tid < HS) {
        // every vector of the pair requested at once, then used
        float kv = 0.f, vv = 0.f;
#pragma unroll 4
        for (int j = 0; j < p.nsplit; ++j) {  // add the projection's k-split slabs in order
            const size_t o = (size_t)j * p.split_stride + off + tid;
            rv += p.r[o];
            kv += p.k[o];
            vv += p.v[o];
        }
        const float av = p.a[off + tid];
        const float decv = p.dec[off + tid];
        const float vf = p.layer == 0 ? 0.f : p.v_first[off + tid];
        const float vgv = p.layer == 0 ? 0.f : p.vg[off + tid];
        const float kk = kv * __low2float(kkka);
        const float ss = sum64(kk * kk, sm.red, 1);
        const float khv = kk / fmaxf(sqrtf(ss), 1e-12f);
        kpv = kv * (1.0f + (av - 1.0f) * __high2float(kkka));
        if (p.layer == 0) {
            vpv = vv;
            p.v_first[off + tid] = vv;
        } else {
            vpv = vv + (vf - vv) * vgv;
        }
        sm.kh[tid] = khv;
        sm.ka[tid] = khv * av;
        sm.dec[tid] = decv;
        sm.kp[tid] = kpv;
        sm.vp[tid] = vpv;
        sm.r[tid] = rv;
    }
    if (tid == 0) sm.ok = mbar_wait(&sm.full, 0u, &sm.ok) ? 1u : 0u;  // sm.ok is 0 while waiting
    __syncthreads();
    const bool got = sm.ok != 0u;
    if (!got) {  // the state copy never arrived: report; nothing is written
        if (tid == 0) atomicOr(p.err, ERR_TIMEOUT);
        return;
    }
    (void)mbar_try_wait(&sm.full, 0u);
    const int rg = tid >> 4, cg = tid & 15;
    const float4 kh = *(const float4 *)&sm.kh[cg * 4];
    const float4 ka = *(const float4 *)&sm.ka[cg * 4];
    const float4 dc = *(const float4 *)&sm.dec[cg * 4];
    const float4 kp = *(const float4 *)&sm.kp[cg * 4];
    const float4 rr = *(const float4 *)&sm.r[cg * 4];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const int i = rg + 8 * q;
        float4 s = ok ? *(const float4 *)&sm.st[i * HS + cg * 4] : make_float4(0.f, 0.f, 0.f, 0.f);
        float sa = s.x * kh.x + s.y * kh.y + s.z * kh.z + s.w * kh.w;
        sa += __shfl_xor_sync(0xffffffffu, sa, 8);
        sa += __shfl_xor_sync(0xffffffffu, sa, 4);
        sa += __shfl_xor_sync(0xffffffffu, sa, 2);
        sa += __shfl_xor_sync(0xffffffffu, sa, 1);
        const float vpi = sm.vp[i];
        s.x = s.x * dc.x - sa * ka.x + vpi * kp.x;
        s.y = s.y * dc.y - sa * ka.y + vpi * kp.y;
        s.z = s.z * dc.z - sa * ka.z + vpi * kp.z;
        s.w = s.w * dc.w - sa * ka.w + vpi * kp.w;
        float y = s.x * rr.x + s.y * rr.y + s.z * rr.z + s.w * rr.w;
        y += __shfl_xor_sync(0xffffffffu, y, 8);
        y += __shfl_xor_sync(0xffffffffu, y, 4);
        y += __shfl_xor_sync(0xffffffffu, y, 2);
        y += __shfl_xor_sync(0xffffffffu, y, 1);
        if (cg == 0) sm.y[i] = y;
        if (ok) __stcs((float4 *)(S + i * HS + cg * 4), s);
    }
    __syncthreads();
    if (tid < HS) {
        const float yv = sm.y[tid];
        // the GroupNorm moments and the bonus sum of the head in one reduction
        Moments m{1.0f, yv, 0.0f};
        float bz = rv * kpv * __low2float(rkg);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const Moments x{__shfl_xor_sync(0xffffffffu, m.n, o), __shfl_xor_sync(0xffffffffu, m.s, o),
                            __shfl_xor_sync(0xffffffffu, m.m2, o)};
            m = merge_moments(m, x);
            bz += __shfl_xor_sync(0xffffffffu, bz, o);
        }
        if ((tid & 31) == 0) {
            float *r4 = sm.red + 4 * (tid >> 5);
            r4[0] = m.n;
            r4[1] = m.s;
            r4[2] = m.m2;
            r4[3] = bz;
        }
        named_bar(1, 64);  // the last use of sm.red: no barrier after the reads
        const Moments t = merge_moments(Moments{sm.red[0], sm.red[1], sm.red[2]}, Moments{sm.red[4], sm.red[5], sm.red[6]});
        const float bonus = sm.red[3] + sm.red[7];
        const float mean = t.s * (1.0f / HS);
        const float dv = yv - mean;
        const float var = t.m2 * (1.0f / HS);
        const float yn = dv * (1.0f / sqrtf(var + 64e-5f)) * __low2float(lnwb) + __high2float(lnwb);
        p.z[off + tid] = __float2half_rn((yn + bonus * vpv) * p.g[off + tid]);
        if (tid == 0) tl_end(p.tl);
    }
}

// ---------------------------------------------------------------------------
// Prefill LayerNorm + token shift: CTA t normalises token t and, for the shift,
// token t-1 again (row 0 takes the slot's shift state), so no CTA waits for
// another.  x is read only; the residual with the slabs added goes to xout.
// CTA 0 also normalises the last token and stores it as the new shift state,
// after it has read the old one.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ln_row(const ElemParams &p, int t, int i0, bool act, const uint4 &w4, const uint4 &b4,
                                       float (&v)[8], float *red) {
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] = 0.0f;
    if (act) {
        ld8f(p.x + (size_t)t * p.d + i0, v);
        if (p.part) add_slabs(v, p.part, p.nsplit, p.split_stride, (size_t)t * p.d + i0);
    }
    ln8(v, act, p.d, w4, b4, red);
}

template <int NMIX>
__global__ void ln_mix_prefill_kernel(const ElemParams p) {
    __shared__ float red[64];
    const int t = blockIdx.x, n = gridDim.x;
    const int i0 = threadIdx.x * 8;
    const bool act = i0 < p.d;
    const int slot = p.single_slot;
    const bool ok = slot >= 0 && slot < p.n_slots;
    uint4 w4 = make_uint4(0, 0, 0, 0), b4 = w4, mu4[NMIX];
    float sh[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float *shp = p.shift + (size_t)(ok ? slot : 0) * p.d + i0;
    if (act) {
        w4 = *reinterpret_cast<const uint4 *>(p.ln_w + i0);
        b4 = *reinterpret_cast<const uint4 *>(p.ln_b + i0);
#pragma unroll
        for (int q = 0; q < NMIX; ++q) mu4[q] = *reinterpret_cast<const uint4 *>(p.mu[q] + i0);
        if (t == 0 && ok) ld8f(shp, sh);
    }
    pdl_wait();
    pdl_launch();
    float v[8];
    if (act) {  // residual of this token for the next phase
        float xv[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) xv[k] = 0.0f;
        ld8f(p.x + (size_t)t * p.d + i0, xv);
        if (p.part) add_slabs(xv, p.part, p.nsplit, p.split_stride, (size_t)t * p.d + i0);
        st8f(p.xout + (size_t)t * p.d + i0, xv);
    }
    ln_row(p, t, i0, act, w4, b4, v, red);
    if (t > 0) ln_row(p, t - 1, i0, act, w4, b4, sh, red);
    if (t == 0 && n > 1) {
        float last[8];
        ln_row(p, n - 1, i0, act, w4, b4, last, red);
        __syncthreads();  // every thread has read the old shift state
        if (act && ok) st8f(shp, last);
    } else if (t == 0) {
        __syncthreads();
        if (act && ok) st8f(shp, v);
    }
    if (!act) return;
#pragma unroll
    for (int q = 0; q < NMIX; ++q) {
        float mu[8], o[8];
        h8_to_f(mu4[q], mu);
#pragma unroll
        for (int k = 0; k < 8; ++k) o[k] = v[k] + (sh[k] - v[k]) * mu[k];
        *reinterpret_cast<uint4 *>(p.xo[q] + (size_t)t * p.d + i0) = f_to_h8(o);
    }
}

// Per (token t, head h), 64 threads (channel j): the WKV vectors.
__global__ void __launch_bounds__(64) wkv_vec_kernel(const WkvSeqParams p) {
    __shared__ float red[2];
    const int h = blockIdx.x, t = blockIdx.y, j = threadIdx.x;
    pdl_wait();
    pdl_launch();
    const int c = h * HS + j;
    const size_t off = (size_t)t * p.d + c;
    float rv = 0.f, kv = 0.f, vv = 0.f;
    for (int s = 0; s < p.nsplit; ++s) {
        const size_t o = (size_t)s * p.split_stride + off;
        rv += p.r[o];
        kv += p.k[o];
        vv += p.v[o];
    }
    const float av = p.a[off];
    const float kk = kv * __half2float(p.k_k[c]);
    const float ss = sum64(kk * kk, red, 1);
    const float khv = kk / fmaxf(sqrtf(ss), 1e-12f);
    const float kpv = kv * (1.0f + (av - 1.0f) * __half2float(p.k_a[c]));
    float vpv;
    if (p.layer == 0) {
        vpv = vv;
        p.v_first[off] = vv;
    } else {
        vpv = vv + (p.v_first[off] - vv) * p.vg[off];
    }
    const float bonus = sum64(rv * kpv * __half2float(p.r_k[c]), red, 1);
    float *vec = p.vec + ((size_t)h * p.vec_rows + t) * (6 * HS) + j;
    vec[0 * HS] = khv;
    vec[1 * HS] = khv * av;
    vec[2 * HS] = p.dec[off];
    vec[3 * HS] = kpv;
    vec[4 * HS] = rv;
    vec[5 * HS] = vpv;
    if (j == 0) p.bonus[(size_t)t * p.H + h] = bonus;
}

// The sequential update of one slot's state over n tokens.  CTA (h, part)
// owns state rows 16*part .. +16 of head h (rows are independent given the
// vectors); thread t: row 16*part + t/8, columns 8*(t%8) .. +8, so the 8
// threads of a row reduce with 3 shuffles.  The vectors of a head are stored
// per token as 6 x 64 contiguous floats, so 32 tokens are one 48 KB block: one
// bulk copy per block, two blocks in flight.
constexpr int WSQ_TB = 32;
struct WsqSmem {
    float vec[2][WSQ_TB][6][HS];
    uint64_t full[2];
    uint32_t stop;
};
__device__ __forceinline__ void wsq_issue(const WkvSeqParams &p, WsqSmem &sm, int h, int blk) {
    const int t0 = blk * WSQ_TB, nb = min(WSQ_TB, p.n - t0);
    const uint32_t bytes = (uint32_t)nb * 6 * HS * 4;
    mbar_expect_tx(&sm.full[blk & 1], bytes);
    bulk_g2s(&sm.vec[blk & 1][0][0][0], p.vec + ((size_t)h * p.vec_rows + t0) * (6 * HS), bytes, &sm.full[blk & 1]);
}
__global__ void __launch_bounds__(128) wkv_seq_kernel(const WkvSeqParams p) {
    extern __shared__ __align__(128) uint8_t wsq_raw[];
    WsqSmem &sm = *reinterpret_cast<WsqSmem *>(wsq_raw);
    const int h = blockIdx.x, part = blockIdx.y, tid = threadIdx.x;
    const int i = 16 * part + (tid >> 3), cb = 8 * (tid & 7);
    const bool ok = p.slot >= 0 && p.slot < p.n_slots;
    float *S = p.wkv + ((size_t)(ok ? p.slot : 0) * p.H + h) * (HS * HS) + (size_t)i * HS + cb;
    float4 s0 = make_float4(0.f, 0.f, 0.f, 0.f), s1 = s0;
    if (ok) {
        s0 = *(const float4 *)S;
        s1 = *(const float4 *)(S + 4);
    }
    const int nblk = (p.n + WSQ_TB - 1) / WSQ_TB;
    if (tid == 0) {
        sm.stop = 0u;
        mbar_init(&sm.full[0], 1);
        mbar_init(&sm.full[1], 1);
        fence_barrier_init();
    }
    __syncthreads();
    pdl_wait();  // the vectors come from the preceding kernel
    pdl_launch();
    if (tid == 0)
        for (int k = 0; k < 2 && k < nblk; ++k) wsq_issue(p, sm, h, k);
    for (int blk = 0; blk < nblk; ++blk) {
        const int t0 = blk * WSQ_TB, nb = min(WSQ_TB, p.n - t0), buf = blk & 1;
        if (tid == 0) sm.stop = mbar_wait(&sm.full[buf], (uint32_t)(blk >> 1) & 1u, &sm.stop) ? 0u : 2u;
        __syncthreads();
        if (sm.stop) {  // a vector block never arrived: report and leave the state as it was
            if (tid == 0) atomicOr(p.err, ERR_TIMEOUT);
            return;
        }
        (void)mbar_try_wait(&sm.full[buf], (uint32_t)(blk >> 1) & 1u);
        for (int tt = 0; tt < nb; ++tt) {
            const float *vv = &sm.vec[buf][tt][0][0];
            const float4 kh0 = *(const float4 *)&vv[0 * HS + cb], kh1 = *(const float4 *)&vv[0 * HS + cb + 4];
            float sa = s0.x * kh0.x + s0.y * kh0.y + s0.z * kh0.z + s0.w * kh0.w + s1.x * kh1.x + s1.y * kh1.y +
                       s1.z * kh1.z + s1.w * kh1.w;
            sa += __shfl_xor_sync(0xffffffffu, sa, 4);
            sa += __shfl_xor_sync(0xffffffffu, sa, 2);
            sa += __shfl_xor_sync(0xffffffffu, sa, 1);
            const float4 ka0 = *(const float4 *)&vv[1 * HS + cb], ka1 = *(const float4 *)&vv[1 * HS + cb + 4];
            const float4 dc0 = *(const float4 *)&vv[2 * HS + cb], dc1 = *(const float4 *)&vv[2 * HS + cb + 4];
            const float4 kp0 = *(const float4 *)&vv[3 * HS + cb], kp1 = *(const float4 *)&vv[3 * HS + cb + 4];
            const float4 r0 = *(const float4 *)&vv[4 * HS + cb], r1 = *(const float4 *)&vv[4 * HS + cb + 4];
            const float vpi = vv[5 * HS + i];
            s0.x = s0.x * dc0.x - sa * ka0.x + vpi * kp0.x;
            s0.y = s0.y * dc0.y - sa * ka0.y + vpi * kp0.y;
            s0.z = s0.z * dc0.z - sa * ka0.z + vpi * kp0.z;
            s0.w = s0.w * dc0.w - sa * ka0.w + vpi * kp0.w;
            s1.x = s1.x * dc1.x - sa * ka1.x + vpi * kp1.x;
            s1.y = s1.y * dc1.y - sa * ka1.y + vpi * kp1.y;
            s1.z = s1.z * dc1.z - sa * ka1.z + vpi * kp1.z;
            s1.w = s1.w * dc1.w - sa * ka1.w + vpi * kp1.w;
            float y = s0.x * r0.x + s0.y * r0.y + s0.z * r0.z + s0.w * r0.w + s1.x * r1.x + s1.y * r1.y +
                      s1.z * r1.z + s1.w * r1.w;
            y += __shfl_xor_sync(0xffffffffu, y, 4);
            y += __shfl_xor_sync(0xffffffffu, y, 2);
            y += __shfl_xor_sync(0xffffffffu, y, 1);
            if ((tid & 7) == 0) p.y[(size_t)(t0 + tt) * p.d + (size_t)h * HS + i] = y;
        }
        __syncthreads();  // buffer fully read
        if (tid == 0 && blk + 2 < nblk) wsq_issue(p, sm, h, blk + 2);
    }
    if (ok) {
        *(float4 *)S = s0;
        *(float4 *)(S + 4) = s1;
    }
}

// Per (token t, head h), 64 threads: z = (GroupNorm(y) * gamma + beta + bonus * vp) * g.
__global__ void __launch_bounds__(64) wkv_gate_kernel(const WkvSeqParams p) {
    __shared__ float red[2];
    const int h = blockIdx.x, t = blockIdx.y, j = threadIdx.x;
    pdl_wait();
    pdl_launch();
    const int c = h * HS + j;
    const size_t off = (size_t)t * p.d + c;
    const float yv = p.y[off];
    const float mean = sum64(yv, red, 1) * (1.0f / HS);
    const float dv = yv - mean;
    const float var = sum64(dv * dv, red, 1) * (1.0f / HS);
    const float yn = dv * (1.0f / sqrtf(var + 64e-5f)) * __half2float(p.lnx_w[c]) + __half2float(p.lnx_b[c]);
    const float vpv = p.vec[((size_t)h * p.vec_rows + t) * (6 * HS) + 5 * HS + j];
    p.z[off] = __float2half_rn((yn + p.bonus[(size_t)t * p.H + h] * vpv) * p.g[off]);
}

// LoRA-down outputs: one CTA per (slot row b, LoRA i); column c of LoRA i is
// the sum of the S partial slabs, passed through the LoRA's activation and
// rounded to fp16.  The LoRA's parameters are picked by constant index (an
// array indexed by a register would be copied to local memory).
__global__ void lora_fin_kernel(const LoraFinParams p) {
    const int b = blockIdx.x, i = blockIdx.y;
    if (threadIdx.x == 0) tl_start(p.tl);
    int r, act;
    const float *part;
    __half *out;
    switch (i) {
        case 0: r = p.r[0], act = p.act[0], part = p.part[0], out = p.out[0]; break;
        case 1: r = p.r[1], act = p.act[1], part = p.part[1], out = p.out[1]; break;
        case 2: r = p.r[2], act = p.act[2], part = p.part[2], out = p.out[2]; break;
        default: r = p.r[3], act = p.act[3], part = p.part[3], out = p.out[3]; break;
    }
    pdl_launch();  // as in ln_mix_kernel: the LoRA-up GEMM may launch and prefetch now
    pdl_wait();
    if (threadIdx.x == 0) tl_release(p.tl);
    const long long stride = (long long)p.bcap * r;
    for (int col = threadIdx.x; col < r; col += blockDim.x) {
        const float *src = part + (size_t)b * r + col;
        float acc = 0.0f;
#pragma unroll 4
        for (int j = 0; j < p.S; ++j) acc += src[(size_t)j * stride];  // the k-split slabs in order
        const float y = act == 1 ? fast_tanh(acc) : (act == 2 ? fast_sigmoid(acc) : acc);
        out[(size_t)b * r + col] = __float2half_rn(y);
    }
    if (threadIdx.x == 0) tl_end(p.tl);
}

// ---------------------------------------------------------------------------
// Slot pool maintenance: reset (zero), copy (recurrent state only) and swap
// (everything a slot holds).
// ---------------------------------------------------------------------------
__global__ void slot_op_kernel(const SlotOpParams p) {
    const size_t per_layer = p.wkv_per_slot + 2 * p.d;
    const size_t total = (size_t)p.L * per_layer + (size_t)p.V;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += stride) {
        float *pa, *pb;
        bool is_occ = false;
        if (e < (size_t)p.L * per_layer) {
            const size_t l = e / per_layer, r = e % per_layer;
            if (r < p.wkv_per_slot) {
                float *base = p.wkv + l * (size_t)p.n_slots * p.wkv_per_slot;
                pa = base + (size_t)p.a * p.wkv_per_slot + r;
                pb = base + (size_t)p.b * p.wkv_per_slot + r;
            } else if (r < p.wkv_per_slot + p.d) {
                float *base = p.shift_att + l * (size_t)p.n_slots * p.d;
                pa = base + (size_t)p.a * p.d + (r - p.wkv_per_slot);
                pb = base + (size_t)p.b * p.d + (r - p.wkv_per_slot);
            } else {
                float *base = p.shift_ffn + l * (size_t)p.n_slots * p.d;
                pa = base + (size_t)p.a * p.d + (r - p.wkv_per_slot - p.d);
                pb = base + (size_t)p.b * p.d + (r - p.wkv_per_slot - p.d);
            }
        } else {
            const size_t r = e - (size_t)p.L * per_layer;
            pa = p.occ + (size_t)p.a * p.V + r;
            pb = p.occ + (size_t)p.b * p.V + r;
            is_occ = true;
        }
        if (p.op == 0) {
            *pa = 0.0f;
        } else if (p.op == 1) {
            *pb = is_occ ? 0.0f : *pa;  // copy state a -> b; b's occurrence counts restart
        } else {
            const float t = *pa;
            *pa = *pb;
            *pb = t;
        }
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        if (p.op == 0) {
            p.ndraw[p.a] = 0ull;
        } else if (p.op == 1) {
            p.ndraw[p.b] = 0ull;
        } else {
            const unsigned long long t = p.ndraw[p.a];
            p.ndraw[p.a] = p.ndraw[p.b];
            p.ndraw[p.b] = t;
            const SampleParamsDev sp = p.params[p.a];
            p.params[p.a] = p.params[p.b];
            p.params[p.b] = sp;
        }
    }
}

static cudaLaunchConfig_t mkcfg(dim3 grid, dim3 block, size_t smem, const LaunchCfg &lc, cudaLaunchAttribute *at) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = lc.stream;
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = lc.pdl ? 1 : 0;
    return cfg;
}

void launch_embed(const ElemParams &p, const LaunchCfg &lc, cudaError_t *e) {
    cudaLaunchAttribute at[1];
    const size_t smem = (size_t)((p.n_slots + 31) / 32) * 4;
    cudaLaunchConfig_t cfg = mkcfg(dim3(p.B), dim3(ln_threads(p.d)), smem, lc, at);
    cudaError_t r = cudaLaunchKernelEx(&cfg, embed_kernel, p);
    if (r != cudaSuccess) *e = r;
}

void launch_ln_mix(const ElemParams &p, int nmix, const LaunchCfg &lc, cudaError_t *e) {
    cudaLaunchAttribute at[1];
    cudaLaunchConfig_t cfg = mkcfg(dim3(p.B), dim3(ln_threads(p.d)), 0, lc, at);
    cudaError_t r = nmix == 6 ? cudaLaunchKernelEx(&cfg, ln_mix_kernel<6>, p) : cudaLaunchKernelEx(&cfg, ln_mix_kernel<1>, p);
    if (r != cudaSuccess) *e = r;
}

void launch_ln_mix_prefill(const ElemParams &p, int nmix, const LaunchCfg &lc, cudaError_t *e) {
    cudaLaunchAttribute at[1];
    cudaLaunchConfig_t cfg = mkcfg(dim3(p.B), dim3(ln_threads(p.d)), 0, lc, at);
    cudaError_t r = nmix == 6 ? cudaLaunchKernelEx(&cfg, ln_mix_prefill_kernel<6>, p)
                              : cudaLaunchKernelEx(&cfg, ln_mix_prefill_kernel<1>, p);
    if (r != cudaSuccess) *e = r;
}

void launch_wkv_prefill(const WkvSeqParams &p, const LaunchCfg &lc, cudaError_t *e) {
    cudaLaunchAttribute at[1];
    cudaLaunchConfig_t c1 = mkcfg(dim3(p.H, p.n), dim3(64), 0, lc, at);
    cudaError_t r = cudaLaunchKernelEx(&c1, wkv_vec_kernel, p);
    if (r == cudaSuccess) {
        r = ensure_smem_attr((const void *)wkv_seq_kernel, (int)sizeof(WsqSmem));
    }
    if (r == cudaSuccess) {
        cudaLaunchConfig_t c2 = mkcfg(dim3(p.H, 4), dim3(128), sizeof(WsqSmem), lc, at);
        r = cudaLaunchKernelEx(&c2, wkv_seq_kernel, p);
    }
    if (r == cudaSuccess) {
        cudaLaunchConfig_t c3 = mkcfg(dim3(p.H, p.n), dim3(64), 0, lc, at);
        r = cudaLaunchKernelEx(&c3, wkv_gate_kernel, p);
    }
    if (r != cudaSuccess) *e = r;
}

void launch_ln_out(const ElemParams &p, const LaunchCfg &lc, cudaError_t *e) {
    cudaLaunchAttribute at[1];
    cudaLaunchConfig_t cfg = mkcfg(dim3(p.B), dim3(ln_threads(p.d)), 0, lc, at);
    cudaError_t r = cudaLaunchKernelEx(&cfg, ln_out_kernel, p);
    if (r != cudaSuccess) *e = r;
}

void launch_wkv(const WkvParams &p, const LaunchCfg &lc, cudaError_t *e) {
    const size_t smem = sizeof(WkvSmem);
    {
        cudaError_t r = ensure_smem_attr((const void *)wkv_kernel, (int)smem);
        if (r != cudaSuccess) {
            *e = r;
            return;
        }
    }
    cudaLaunchAttribute at[1];
    cudaLaunchConfig_t cfg = mkcfg(dim3(p.H, p.B), dim3(WKV_THREADS), smem, lc, at);
    cudaError_t r = cudaLaunchKernelEx(&cfg, wkv_kernel, p);
    if (r != cudaSuccess) *e = r;
}

void launch_lora_fin(const LoraFinParams &p, const LaunchCfg &lc, cudaError_t *e) {
    cudaLaunchAttribute at[1];
    cudaLaunchConfig_t cfg = mkcfg(dim3(p.B, 4), dim3(128), 0, lc, at);
    cudaError_t r = cudaLaunchKernelEx(&cfg, lora_fin_kernel, p);
    if (r != cudaSuccess) *e = r;
}

void launch_slot_op(const SlotOpParams &p, cudaStream_t s, cudaError_t *e) {
    slot_op_kernel<<<304, 256, 0, s>>>(p);
    cudaError_t r = cudaGetLastError();
    if (r != cudaSuccess) *e = r;
}

}  // namespace rk
