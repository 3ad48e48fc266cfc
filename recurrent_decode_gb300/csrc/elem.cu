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

constexpr int LN_THREADS = 256;
constexpr int LN_MAXV = 32;  // d <= 8192

// Sum over the CTA (blockDim = LN_THREADS).  `red` holds 32 floats.
__device__ __forceinline__ float block_sum(float v, float *red) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    v = warp_sum(v);
    __syncthreads();
    if (lane == 0) red[w] = v;
    __syncthreads();
    float t = 0.0f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) t += red[i];
    return t;
}

// LayerNorm of the values v[j] = x[tid + j*blockDim] (j < cnt, d values in all),
// in place: (x - mean) / sqrt(var + eps) * w + b with biased variance.
__device__ __forceinline__ void block_layernorm(float (&v)[LN_MAXV], int d, const __half *w, const __half *b,
                                                float *red) {
    const int cnt = (d + LN_THREADS - 1) / LN_THREADS;
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < LN_MAXV; ++j)
        if (j < cnt && threadIdx.x + j * LN_THREADS < d) s += v[j];
    const float mean = block_sum(s, red) / (float)d;
    float q = 0.0f;
#pragma unroll
    for (int j = 0; j < LN_MAXV; ++j)
        if (j < cnt && threadIdx.x + j * LN_THREADS < d) {
            float t = v[j] - mean;
            q += t * t;
        }
    const float var = block_sum(q, red) / (float)d;
    const float rs = 1.0f / sqrtf(var + 1e-5f);
#pragma unroll
    for (int j = 0; j < LN_MAXV; ++j) {
        const int i = threadIdx.x + j * LN_THREADS;
        if (j < cnt && i < d) v[j] = (v[j] - mean) * rs * __half2float(w[i]) + __half2float(b[i]);
    }
}

// x[b] = LN0(emb[token[b]]).  Also validates the step's slots and tokens:
// range errors are latched and the row falls back to token 0; CTA 0 looks for
// repeated slots with a bitmap in shared memory.
__global__ void __launch_bounds__(LN_THREADS) embed_kernel(const ElemParams p) {
    extern __shared__ uint32_t bitmap[];
    __shared__ float red[32];
    pdl_wait();
    pdl_launch();
    const int b = blockIdx.x;
    const int slot = p.slots[b];
    int tok = p.tokens[b];
    if (threadIdx.x == 0) {
        if (slot < 0 || slot >= p.n_slots) atomicOr(p.err, ERR_SLOT);
        if (tok < 0 || tok >= p.V) atomicOr(p.err, ERR_TOKEN);
    }
    if (tok < 0 || tok >= p.V) tok = 0;
    const __half *e = p.emb + (size_t)tok * p.d;
    float v[LN_MAXV];
    const int cnt = (p.d + LN_THREADS - 1) / LN_THREADS;
#pragma unroll
    for (int j = 0; j < LN_MAXV; ++j) {
        const int i = threadIdx.x + j * LN_THREADS;
        v[j] = (j < cnt && i < p.d) ? __half2float(e[i]) : 0.0f;
    }
    block_layernorm(v, p.d, p.ln_w, p.ln_b, red);
    float *xr = p.x + (size_t)b * p.d;
#pragma unroll
    for (int j = 0; j < LN_MAXV; ++j) {
        const int i = threadIdx.x + j * LN_THREADS;
        if (j < cnt && i < p.d) xr[i] = v[j];
    }
    if (b == 0) {
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
// nmix = 6 for the time mix (r, w, k, v, a, g), 1 for the channel mix.
__global__ void __launch_bounds__(LN_THREADS) ln_mix_kernel(const ElemParams p, int nmix) {
    __shared__ float red[32];
    const int b = blockIdx.x;
    const int slot = p.slots[b];
    const bool ok = slot >= 0 && slot < p.n_slots;
    pdl_wait();
    pdl_launch();
    const float *xr = p.x + (size_t)b * p.d;
    float v[LN_MAXV];
    const int cnt = (p.d + LN_THREADS - 1) / LN_THREADS;
#pragma unroll
    for (int j = 0; j < LN_MAXV; ++j) {
        const int i = threadIdx.x + j * LN_THREADS;
        v[j] = (j < cnt && i < p.d) ? xr[i] : 0.0f;
    }
    block_layernorm(v, p.d, p.ln_w, p.ln_b, red);
    float *sh = p.shift + (size_t)(ok ? slot : 0) * p.d;
#pragma unroll
    for (int j = 0; j < LN_MAXV; ++j) {
        const int i = threadIdx.x + j * LN_THREADS;
        if (j < cnt && i < p.d) {
            const float xl = v[j];
            const float prev = ok ? sh[i] : 0.0f;
            const float dlt = prev - xl;
            for (int q = 0; q < nmix; ++q)
                p.xo[q][(size_t)b * p.d + i] = __float2half_rn(xl + dlt * __half2float(p.mu[q][i]));
            if (ok) sh[i] = xl;
        }
    }
}

// xo[0][b] = fp16(LN_out(x[b])): the input of the head projection.
__global__ void __launch_bounds__(LN_THREADS) ln_out_kernel(const ElemParams p) {
    __shared__ float red[32];
    const int b = blockIdx.x;
    pdl_wait();
    pdl_launch();
    const float *xr = p.x + (size_t)b * p.d;
    float v[LN_MAXV];
    const int cnt = (p.d + LN_THREADS - 1) / LN_THREADS;
#pragma unroll
    for (int j = 0; j < LN_MAXV; ++j) {
        const int i = threadIdx.x + j * LN_THREADS;
        v[j] = (j < cnt && i < p.d) ? xr[i] : 0.0f;
    }
    block_layernorm(v, p.d, p.ln_w, p.ln_b, red);
#pragma unroll
    for (int j = 0; j < LN_MAXV; ++j) {
        const int i = threadIdx.x + j * LN_THREADS;
        if (j < cnt && i < p.d) p.xo[0][(size_t)b * p.d + i] = __float2half_rn(v[j]);
    }
}

// ---------------------------------------------------------------------------
// WKV7: one CTA per (head h, slot row b), 256 threads.  Thread t holds state
// rows i0 + 16q (q = 0..3, i0 = t / 16) at columns 4(t % 16) .. +3, so every
// 16-lane group owns whole rows and the row reductions are 4 shuffles.
//   kh = normalize(k * k_k), kp = k * (1 + (a - 1) * k_a),
//   vp = v (layer 0, also stored as v_first) or v + (v_first - v) * vg,
//   S[i][j] <- S[i][j] dec_j - (sum_m S[i][m] kh_m) kh_j a_j + vp_i kp_j,
//   y_i = sum_j S[i][j] r_j,
//   z = (GroupNorm(y) * gamma + beta + (sum_j r_j kp_j r_k_j) vp) * g  -> fp16.
// The state tile (16 KB) is fetched before the dependency wait: only this
// kernel (one layer, one step earlier) writes it.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float sum64(float v, float *s2, int barid) {
    v = warp_sum(v);
    if ((threadIdx.x & 31) == 0) s2[threadIdx.x >> 5] = v;
    named_bar(barid, 64);
    const float t = s2[0] + s2[1];
    named_bar(barid, 64);
    return t;
}

__global__ void __launch_bounds__(256) wkv_kernel(const WkvParams p) {
    __shared__ __align__(16) float s_kh[HS], s_ka[HS], s_dec[HS], s_kp[HS], s_vp[HS], s_r[HS], s_y[HS];
    __shared__ float s_red[4];
    const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
    const int slot = p.slots[b];
    const bool ok = slot >= 0 && slot < p.n_slots;
    float *S = p.wkv + ((size_t)(ok ? slot : 0) * p.H + h) * (HS * HS);
    const int i0 = tid >> 4, cg = tid & 15;
    float4 st[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
        st[q] = ok ? __ldcs((const float4 *)(S + (i0 + 16 * q) * HS + cg * 4)) : make_float4(0.f, 0.f, 0.f, 0.f);
    pdl_wait();
    pdl_launch();

    const size_t off = (size_t)b * p.d + (size_t)h * HS;
    float kk = 0.f, kv = 0.f, av = 0.f, vv = 0.f;
    if (tid < HS) {
        const int c = h * HS + tid;
        kv = p.k[off + tid];
        av = p.a[off + tid];
        vv = p.v[off + tid];
        kk = kv * __half2float(p.k_k[c]);
        const float ss = sum64(kk * kk, s_red, 1);
        const float nrm = fmaxf(sqrtf(ss), 1e-12f);
        const float khv = kk / nrm;
        const float kpv = kv * (1.0f + (av - 1.0f) * __half2float(p.k_a[c]));
        float vpv;
        if (p.layer == 0) {
            vpv = vv;
            p.v_first[off + tid] = vv;
        } else {
            const float vf = p.v_first[off + tid];
            vpv = vv + (vf - vv) * p.vg[off + tid];
        }
        s_kh[tid] = khv;
        s_ka[tid] = khv * av;
        s_dec[tid] = p.dec[off + tid];
        s_kp[tid] = kpv;
        s_vp[tid] = vpv;
        s_r[tid] = p.r[off + tid];
    }
    __syncthreads();
    const float4 kh = *(const float4 *)&s_kh[cg * 4];
    const float4 ka = *(const float4 *)&s_ka[cg * 4];
    const float4 dc = *(const float4 *)&s_dec[cg * 4];
    const float4 kp = *(const float4 *)&s_kp[cg * 4];
    const float4 rr = *(const float4 *)&s_r[cg * 4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int i = i0 + 16 * q;
        float4 s = st[q];
        float sa = s.x * kh.x + s.y * kh.y + s.z * kh.z + s.w * kh.w;
        sa += __shfl_xor_sync(0xffffffffu, sa, 8);
        sa += __shfl_xor_sync(0xffffffffu, sa, 4);
        sa += __shfl_xor_sync(0xffffffffu, sa, 2);
        sa += __shfl_xor_sync(0xffffffffu, sa, 1);
        const float vpi = s_vp[i];
        s.x = s.x * dc.x - sa * ka.x + vpi * kp.x;
        s.y = s.y * dc.y - sa * ka.y + vpi * kp.y;
        s.z = s.z * dc.z - sa * ka.z + vpi * kp.z;
        s.w = s.w * dc.w - sa * ka.w + vpi * kp.w;
        float y = s.x * rr.x + s.y * rr.y + s.z * rr.z + s.w * rr.w;
        y += __shfl_xor_sync(0xffffffffu, y, 8);
        y += __shfl_xor_sync(0xffffffffu, y, 4);
        y += __shfl_xor_sync(0xffffffffu, y, 2);
        y += __shfl_xor_sync(0xffffffffu, y, 1);
        if (cg == 0) s_y[i] = y;
        if (ok) __stcs((float4 *)(S + i * HS + cg * 4), s);
    }
    __syncthreads();
    if (tid < HS) {
        const int c = h * HS + tid;
        const float yv = s_y[tid];
        const float mean = sum64(yv, s_red, 1) * (1.0f / HS);
        const float dv = yv - mean;
        const float var = sum64(dv * dv, s_red, 1) * (1.0f / HS);
        const float yn = dv * (1.0f / sqrtf(var + 64e-5f)) * __half2float(p.lnx_w[c]) + __half2float(p.lnx_b[c]);
        const float bonus = sum64(s_r[tid] * s_kp[tid] * __half2float(p.r_k[c]), s_red, 1);
        const float zv = (yn + bonus * s_vp[tid]) * p.g[off + tid];
        p.z[off + tid] = __float2half_rn(zv);
    }
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
    cudaLaunchConfig_t cfg = mkcfg(dim3(p.B), dim3(LN_THREADS), smem, lc, at);
    cudaError_t r = cudaLaunchKernelEx(&cfg, embed_kernel, p);
    if (r != cudaSuccess) *e = r;
}

void launch_ln_mix(const ElemParams &p, int nmix, const LaunchCfg &lc, cudaError_t *e) {
    cudaLaunchAttribute at[1];
    cudaLaunchConfig_t cfg = mkcfg(dim3(p.B), dim3(LN_THREADS), 0, lc, at);
    cudaError_t r = cudaLaunchKernelEx(&cfg, ln_mix_kernel, p, nmix);
    if (r != cudaSuccess) *e = r;
}

void launch_ln_out(const ElemParams &p, const LaunchCfg &lc, cudaError_t *e) {
    cudaLaunchAttribute at[1];
    cudaLaunchConfig_t cfg = mkcfg(dim3(p.B), dim3(LN_THREADS), 0, lc, at);
    cudaError_t r = cudaLaunchKernelEx(&cfg, ln_out_kernel, p);
    if (r != cudaSuccess) *e = r;
}

void launch_wkv(const WkvParams &p, const LaunchCfg &lc, cudaError_t *e) {
    cudaLaunchAttribute at[1];
    cudaLaunchConfig_t cfg = mkcfg(dim3(p.H, p.B), dim3(256), 0, lc, at);
    cudaError_t r = cudaLaunchKernelEx(&cfg, wkv_kernel, p);
    if (r != cudaSuccess) *e = r;
}

void launch_slot_op(const SlotOpParams &p, cudaStream_t s, cudaError_t *e) {
    slot_op_kernel<<<304, 256, 0, s>>>(p);
    cudaError_t r = cudaGetLastError();
    if (r != cudaSuccess) *e = r;
}

}  // namespace rk
