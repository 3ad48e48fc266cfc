// persist.cu -- the whole decode step as one persistent kernel.
//
// The step is a chain of small dependent operations per layer (the pages' T=1
// fused branch, "RWKV 批量推理中 Prefill 的正确打开方式" §三, runs them as separate
// kernels).  Launched one after another, each operation pays its own fill,
// drain and launch gaps, and the HBM stream stops at every boundary.  Here one
// cooperative grid (one CTA per SM) runs every layer; the two byte streams that
// do not depend on the step's activations -- the fp16 weight tiles and the fp32
// recurrent states of the slots -- are fetched into a ring of shared-memory
// stages as fast as the ring drains, across operation boundaries, while the
// activation operands are fetched once the operation that produces them has
// signalled completion through a global counter.
//
// Roles (192 threads):
//   warp 0 lane 0  producer: weight tiles (TMA), slot states (bulk copies) and,
//                  when their producer phase is complete, activation boxes (TMA)
//   warp 1         TMEM owner; lane 0 issues tcgen05.mma into two accumulators
//   warps 2-5      128 "row" threads: GEMM epilogues (TMEM -> registers ->
//                  outputs), LayerNorm + token-shift rows, the WKV7 update of
//                  (slot, head) pairs from the ring, GroupNorm / bonus / gate.
// Phases of layer l, each signalling counter cnt[l * 8 + phase]:
//   LN1 (rows) -> G1 r,k,v + LoRA-down -> G2 LoRA-up -> WKV (slot, head pairs)
//   -> G3 output proj -> LN2 (rows) -> G4 key + ReLU^2 -> G5 value
// then LN_out (rows) and the head projection.  Split-K items either store raw
// partial slabs that the consuming row phase adds in slab order (G3, G5), or
// the tile's last split (by a per-tile counter) adds the slabs in order and
// applies the epilogue (G1, G4, head).  Every wait is bounded by %globaltimer
// and a shared abort word, after which the kernel latches ERR_TIMEOUT and
// returns.
#include "internal.cuh"

namespace rk {
namespace {

constexpr int PK_THREADS = 192;
constexpr int NROW = 128;  // row threads (warps 2-5)
constexpr uint32_t TILE_B = GEMM_TILE_M * GEMM_TILE_K * 2;  // 16 KB weight tile
constexpr uint32_t PAIR_B = HS * HS * 4;                     // 16 KB state of one (slot, head)
constexpr int PH_HEAD = 8;                                   // producer / MMA phase id of the head
constexpr int BAR_ROW = 1;                                   // named barrier of the 128 row threads
constexpr int BAR_HALF = 2;                                  // named barrier of row threads 0..63

enum { PH_LN1 = 0, PH_G1, PH_G2, PH_WKV, PH_G3, PH_LN2, PH_G4, PH_G5 };

struct SmemTail {
    PkGemm g[PKG_COUNT];
    alignas(16) float vkh[2][HS];   // per half of the row threads: one (slot, head) pair each
    alignas(16) float vka[2][HS];
    alignas(16) float vdec[2][HS];
    alignas(16) float vkp[2][HS];
    alignas(16) float vr[2][HS];
    float red[8];
    uint32_t tmem_base;
    uint32_t flag;
    uint32_t state_done;  // state stages released by the row threads (MMA-side ordering)
};

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void mbar_expect_tx_noarrive(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

__device__ __forceinline__ bool aborted(const uint32_t *abort_flag) {
    return *(volatile const uint32_t *)abort_flag != 0u;
}
__device__ __forceinline__ void give_up(const PkParams &p) {
    atomicExch(p.abort_flag, 1u);
    atomicOr(p.err, ERR_TIMEOUT);
}
// Record the first wait that gave up: code (1 producer, 2 MMA accumulator,
// 3 MMA stage, 4 counter, 5 row stage / accumulator), CTA and four details.
__device__ void note(const PkParams &p, uint32_t code, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    if (atomicCAS(p.diag, 0u, code) == 0u) {
        p.diag[1] = blockIdx.x;
        p.diag[2] = a;
        p.diag[3] = b;
        p.diag[4] = c;
        p.diag[5] = d;
        __threadfence();
    }
}
// Bounded wait until *c >= target.
__device__ bool wait_count(const uint32_t *c, uint32_t target, const uint32_t *abort_flag) {
    if (ld_acquire(c) >= target) return true;
    const uint64_t t0 = gtimer();
    for (uint32_t it = 1;; ++it) {
        if (ld_acquire(c) >= target) return true;
        __nanosleep(64);
        if ((it & 31u) == 0) {
            if (aborted(abort_flag)) return false;
            if (gtimer() - t0 > WAIT_LIMIT_NS) return false;
        }
    }
}
// Waits of the single-thread roles back off with __nanosleep once the first
// polls fail: a spinning warp takes issue slots from the row warps that share
// its scheduler.
__device__ bool pk_mbar_wait(uint64_t *bar, uint32_t parity, const uint32_t *abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = gtimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if (it > 4) __nanosleep(64);
        if ((it & 31u) == 0) {
            if (aborted(abort_flag)) return false;
            if (gtimer() - t0 > WAIT_LIMIT_NS) return false;
        }
    }
}
__device__ __forceinline__ void signal_count(uint32_t *c, uint32_t n) {
    __threadfence();
    atomicAdd(c, n);
}

__device__ __forceinline__ int first_of(int c, int G, int n) { return (int)(((long long)c * n) / G); }

struct PItem {
    int s, tile, split, kb0, kb1;
};
__device__ __forceinline__ PItem locate(const PkGemm &g, int i, int kbs) {
    int s = 0;
    while (s + 1 < g.nseg && i >= g.seg[s + 1].item0) ++s;
    const PkSeg &sg = g.seg[s];
    const int local = i - sg.item0;
    PItem it;
    it.s = s;
    it.tile = local / sg.S;
    it.split = local - it.tile * sg.S;
    const int np = sg.kb / kbs;
    it.kb0 = (int)(((long long)it.split * np) / sg.S) * kbs;
    it.kb1 = (int)(((long long)(it.split + 1) * np) / sg.S) * kbs;
    return it;
}
__device__ __forceinline__ int gemm_of(int l, int ph) {
    switch (ph) {
        case PH_G1: return l ? PKG_G1 : PKG_G1_0;
        case PH_G2: return l ? PKG_G2 : PKG_G2_0;
        case PH_G3: return PKG_G3;
        case PH_G4: return PKG_G4;
        case PH_G5: return PKG_G5;
        default: return PKG_HEAD;
    }
}
// Ring stages of this CTA's items of one GEMM phase.
__device__ int gemm_stages(const PkGemm &g, int c, int G, int kbs) {
    int n = 0;
    for (int i = first_of(c, G, g.nitems), e = first_of(c + 1, G, g.nitems); i < e; ++i) {
        const PItem it = locate(g, i, kbs);
        n += (it.kb1 - it.kb0) / kbs;
    }
    return n;
}
__device__ __forceinline__ int wkv_stages(int c, int G, int npairs, int kbs) {
    const int n = first_of(c + 1, G, npairs) - first_of(c, G, npairs);
    return (n + kbs - 1) / kbs;
}

// ---------------------------------------------------------------------------
// Stage cursor: walks this CTA's ring stages in issue order.
// ---------------------------------------------------------------------------
struct Cursor {
    int l, ph;      // layer, phase (PH_G1.., PH_WKV, or PH_HEAD with l == L)
    int i, iend;    // GEMM item or WKV pair range
    int kb, kb1;    // current k-block range of the GEMM item
    int s, tile;
    bool done;
};

__device__ void cur_enter(Cursor &u, const PkParams &p, const SmemTail &t, int c, int G);

__device__ void cur_next_phase(Cursor &u, const PkParams &p, const SmemTail &t, int c, int G) {
    if (u.ph == PH_HEAD) {
        u.done = true;
        return;
    }
    if (u.ph == PH_G5) {
        if (u.l + 1 < p.L) {
            ++u.l;
            u.ph = PH_G1;
        } else if (p.head) {
            u.l = p.L;
            u.ph = PH_HEAD;
        } else {
            u.done = true;
            return;
        }
    } else {
        u.ph = (u.ph == PH_G1) ? PH_G2 : (u.ph == PH_G2) ? PH_WKV : (u.ph == PH_WKV) ? PH_G3 : (u.ph == PH_G3) ? PH_G4 : PH_G5;
    }
    cur_enter(u, p, t, c, G);
}

__device__ void cur_load_item(Cursor &u, const PkParams &p, const SmemTail &t) {
    const PItem it = locate(t.g[gemm_of(u.l, u.ph)], u.i, p.kbs);
    u.s = it.s;
    u.tile = it.tile;
    u.kb = it.kb0;
    u.kb1 = it.kb1;
}

// Position the cursor on the first non-empty stage at or after the current phase.
__device__ void cur_enter(Cursor &u, const PkParams &p, const SmemTail &t, int c, int G) {
    for (;;) {
        if (u.ph == PH_WKV) {
            const int n = p.B * p.H;
            u.i = first_of(c, G, n);
            u.iend = first_of(c + 1, G, n);
            if (u.i < u.iend) return;
        } else {
            const PkGemm &g = t.g[gemm_of(u.l, u.ph)];
            u.i = first_of(c, G, g.nitems);
            u.iend = first_of(c + 1, G, g.nitems);
            for (; u.i < u.iend; ++u.i) {
                cur_load_item(u, p, t);
                if (u.kb < u.kb1) return;
            }
        }
        // empty phase: move on
        if (u.ph == PH_HEAD) {
            u.done = true;
            return;
        }
        if (u.ph == PH_G5) {
            if (u.l + 1 < p.L) {
                ++u.l;
                u.ph = PH_G1;
            } else if (p.head) {
                u.l = p.L;
                u.ph = PH_HEAD;
            } else {
                u.done = true;
                return;
            }
        } else {
            u.ph = (u.ph == PH_G1) ? PH_G2 : (u.ph == PH_G2) ? PH_WKV : (u.ph == PH_WKV) ? PH_G3 : (u.ph == PH_G3) ? PH_G4 : PH_G5;
        }
    }
}

__device__ void cur_begin(Cursor &u, const PkParams &p, const SmemTail &t, int c, int G) {
    u.l = 0;
    u.ph = PH_G1;
    u.done = false;
    cur_enter(u, p, t, c, G);
}

// Advance by one stage.
__device__ void cur_next(Cursor &u, const PkParams &p, const SmemTail &t, int c, int G) {
    if (u.ph == PH_WKV) {
        u.i += p.kbs;
        if (u.i < u.iend) return;
        cur_next_phase(u, p, t, c, G);
        return;
    }
    u.kb += p.kbs;
    if (u.kb < u.kb1) return;
    for (++u.i; u.i < u.iend; ++u.i) {
        cur_load_item(u, p, t);
        if (u.kb < u.kb1) return;
    }
    cur_next_phase(u, p, t, c, G);
}

// Counter and target that make the activations of a GEMM phase ready.
__device__ __forceinline__ void x_dep(const PkParams &p, const SmemTail &t, int l, int ph, const uint32_t **cnt,
                                      uint32_t *target) {
    switch (ph) {
        case PH_G1: *cnt = p.cnt + l * PK_NPH + PH_LN1; *target = (uint32_t)p.B; break;
        case PH_G2: *cnt = p.cnt + l * PK_NPH + PH_G1; *target = (uint32_t)t.g[gemm_of(l, PH_G1)].nitems; break;
        case PH_G3: *cnt = p.cnt + l * PK_NPH + PH_WKV; *target = (uint32_t)(p.B * p.H); break;
        case PH_G4: *cnt = p.cnt + l * PK_NPH + PH_LN2; *target = (uint32_t)p.B; break;
        case PH_G5: *cnt = p.cnt + l * PK_NPH + PH_G4; *target = (uint32_t)t.g[PKG_G4].nitems; break;
        default: *cnt = p.cnt + p.L * PK_NPH; *target = (uint32_t)p.B; break;
    }
}

// ---------------------------------------------------------------------------
// Epilogue stores.  v[q] is the fp32 result for slot row cb + q of weight row n.
// ---------------------------------------------------------------------------

template <int KIND>
__device__ __forceinline__ void store_final(const PkSeg &sg, int n, int cb, int nq, const float (&v)[32], float bias) {
    const size_t ldo = (size_t)sg.ldo;
    if (KIND == EPI_F32 || KIND == EPI_DECAY || KIND == EPI_SIGMOID_BIAS) {
        float *out = (float *)sg.out + (size_t)cb * ldo + n;
#pragma unroll
        for (int q = 0; q < 32; ++q) {
            float y = v[q];
            if (KIND == EPI_DECAY) y = rwkv_decay(bias + y);
            if (KIND == EPI_SIGMOID_BIAS) y = fast_sigmoid(bias + y);
            if (q < nq) out[(size_t)q * ldo] = y;
        }
    } else {
        __half *out = (__half *)sg.out + (size_t)cb * ldo + n;
#pragma unroll
        for (int q = 0; q < 32; ++q) {
            float y = v[q];
            if (KIND == EPI_F16_TANH) y = fast_tanh(y);
            if (KIND == EPI_F16_SIGMOID) y = fast_sigmoid(y);
            if (KIND == EPI_RELU2) {
                y = fmaxf(y, 0.0f);
                y = y * y;
            }
            if (q < nq) out[(size_t)q * ldo] = __float2half_rn(y);
        }
    }
}
__device__ __forceinline__ void store_partial(const PkSeg &sg, int split, int n, int cb, int nq, const float (&v)[32]) {
    const size_t ldo = (size_t)sg.ldo;
    float *out = sg.part + (size_t)split * sg.split_stride + (size_t)cb * ldo + n;
#pragma unroll
    for (int q = 0; q < 32; ++q)
        if (q < nq) out[(size_t)q * ldo] = v[q];
}

// Read one 32-column chunk of the accumulator (zeros when nothing was issued).
__device__ __forceinline__ void acc_chunk(uint32_t taddr, int cb, int npad, bool valid, float (&v)[32]) {
    if (valid) {
        if (cb + 32 <= npad) {
            tmem_ld32(taddr + (uint32_t)cb, v);
        } else {
            float h[16];
            tmem_ld16(taddr + (uint32_t)cb, h);
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                v[q] = h[q];
                v[q + 16] = 0.0f;
            }
        }
    } else {
#pragma unroll
        for (int q = 0; q < 32; ++q) v[q] = 0.0f;
    }
}

template <int KIND>
__device__ __forceinline__ void epi_direct(const PkSeg &sg, uint32_t taddr, bool valid, int n, int npad, int B, float bias) {
    const bool live = n < sg.rows;
    for (int cb = 0; cb < npad; cb += 32) {
        float v[32];
        acc_chunk(taddr, cb, npad, valid, v);
        if (live) store_final<KIND>(sg, n, cb, min(32, B - cb), v, bias);
    }
}
__device__ __forceinline__ void epi_partial(const PkSeg &sg, uint32_t taddr, bool valid, int n, int split, int npad, int B) {
    const bool live = n < sg.rows;
    for (int cb = 0; cb < npad; cb += 32) {
        float v[32];
        acc_chunk(taddr, cb, npad, valid, v);
        if (live) store_partial(sg, split, n, cb, min(32, B - cb), v);
    }
}
// The tile's last split: out = epilogue(sum of the S slabs in slab order).
// Each slab's 32 (or 64) loads per thread are issued together.
template <int KIND>
__device__ __forceinline__ void epi_fixup(const PkSeg &sg, int n, int B, float bias) {
    if (n >= sg.rows) return;
    for (int cb = 0; cb < B; cb += 64) {
        const int nq0 = min(32, B - cb), nq1 = min(32, B - cb - 32);
        float v0[32], v1[32];
#pragma unroll
        for (int q = 0; q < 32; ++q) {
            v0[q] = 0.0f;
            v1[q] = 0.0f;
        }
        for (int j = 0; j < sg.S; ++j) {
            const float *src = sg.part + (size_t)j * sg.split_stride + (size_t)cb * sg.ldo + n;
            float t0[32], t1[32];
#pragma unroll
            for (int q = 0; q < 32; ++q) {
                t0[q] = q < nq0 ? __ldcg(src + (size_t)q * sg.ldo) : 0.0f;
                t1[q] = q < nq1 ? __ldcg(src + (size_t)(q + 32) * sg.ldo) : 0.0f;
            }
#pragma unroll
            for (int q = 0; q < 32; ++q) {
                v0[q] += t0[q];
                v1[q] += t1[q];
            }
        }
        store_final<KIND>(sg, n, cb, nq0, v0, bias);
        if (nq1 > 0) store_final<KIND>(sg, n, cb + 32, nq1, v1, bias);
    }
}
template <int KIND>
__device__ __forceinline__ void epi_kind(const PkSeg &sg, bool fixup, uint32_t taddr, bool valid, int n, int npad, int B, float bias) {
    if (fixup)
        epi_fixup<KIND>(sg, n, B, bias);
    else
        epi_direct<KIND>(sg, taddr, valid, n, npad, B, bias);
}
__device__ __forceinline__ void epi_final(const PkSeg &sg, bool fixup, uint32_t taddr, bool valid, int n, int npad, int B, float bias) {
    switch (sg.epi) {
        case EPI_F32: epi_kind<EPI_F32>(sg, fixup, taddr, valid, n, npad, B, bias); break;
        case EPI_F16: epi_kind<EPI_F16>(sg, fixup, taddr, valid, n, npad, B, bias); break;
        case EPI_F16_TANH: epi_kind<EPI_F16_TANH>(sg, fixup, taddr, valid, n, npad, B, bias); break;
        case EPI_F16_SIGMOID: epi_kind<EPI_F16_SIGMOID>(sg, fixup, taddr, valid, n, npad, B, bias); break;
        case EPI_DECAY: epi_kind<EPI_DECAY>(sg, fixup, taddr, valid, n, npad, B, bias); break;
        case EPI_SIGMOID_BIAS: epi_kind<EPI_SIGMOID_BIAS>(sg, fixup, taddr, valid, n, npad, B, bias); break;
        case EPI_RELU2: epi_kind<EPI_RELU2>(sg, fixup, taddr, valid, n, npad, B, bias); break;
        default: break;
    }
}

// ---------------------------------------------------------------------------
// Row helpers for the 128 row threads (8 consecutive elements per chunk,
// chunks et, et + 128, ...; d <= 4096).
// ---------------------------------------------------------------------------
constexpr int MAXCH = 4;

__device__ __forceinline__ void h8f(const uint4 &u, float (&f)[8]) {
    const __half2 *h = reinterpret_cast<const __half2 *>(&u);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 t = __half22float2(h[k]);
        f[2 * k] = t.x;
        f[2 * k + 1] = t.y;
    }
}
__device__ __forceinline__ uint4 fh8(const float (&f)[8]) {
    uint4 u;
    __half2 *h = reinterpret_cast<__half2 *>(&u);
#pragma unroll
    for (int k = 0; k < 4; ++k) h[k] = __floats2half2_rn(f[2 * k], f[2 * k + 1]);
    return u;
}
__device__ __forceinline__ void ld8cg(const float *p, float (&f)[8]) {
    const float4 a = __ldcg(reinterpret_cast<const float4 *>(p)), b = __ldcg(reinterpret_cast<const float4 *>(p + 4));
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}
__device__ __forceinline__ void st8(float *p, const float (&f)[8]) {
    *reinterpret_cast<float4 *>(p) = make_float4(f[0], f[1], f[2], f[3]);
    *reinterpret_cast<float4 *>(p + 4) = make_float4(f[4], f[5], f[6], f[7]);
}

__device__ __forceinline__ float row_sum(float v, float *red, int et) {
    v = warp_sum(v);
    named_bar(BAR_ROW, NROW);
    if ((et & 31) == 0) red[et >> 5] = v;
    named_bar(BAR_ROW, NROW);
    return red[0] + red[1] + red[2] + red[3];
}

// LayerNorm of the row held in v (inactive chunks hold zeros).
__device__ __forceinline__ void row_ln(float (&v)[MAXCH][8], int d, int et, const __half *w, const __half *b, float *red) {
    float s = 0.0f;
#pragma unroll
    for (int m = 0; m < MAXCH; ++m)
#pragma unroll
        for (int k = 0; k < 8; ++k) s += v[m][k];
    const float mean = row_sum(s, red, et) / (float)d;
    float q = 0.0f;
#pragma unroll
    for (int m = 0; m < MAXCH; ++m) {
        const int i0 = (et + NROW * m) * 8;
        if (i0 < d)
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float t = v[m][k] - mean;
                q += t * t;
            }
    }
    const float var = row_sum(q, red, et) / (float)d;
    const float rs = 1.0f / sqrtf(var + 1e-5f);
#pragma unroll
    for (int m = 0; m < MAXCH; ++m) {
        const int i0 = (et + NROW * m) * 8;
        if (i0 < d) {
            float wf[8], bf[8];
            h8f(*reinterpret_cast<const uint4 *>(w + i0), wf);
            h8f(*reinterpret_cast<const uint4 *>(b + i0), bf);
#pragma unroll
            for (int k = 0; k < 8; ++k) v[m][k] = (v[m][k] - mean) * rs * wf[k] + bf[k];
        }
    }
}


// Token-shift mixes of a normalised row: out_q = fp16(xl + (shift - xl) * mu_q),
// shift <- xl.  The shift state and the NMIX mix vectors of a chunk are loaded
// together.
template <int NMIX>
__device__ __forceinline__ void mix_out(const PkParams &p, const float (&v)[MAXCH][8], float *shift, bool ok, int b,
                                        size_t lo, int et) {
    const int d = p.d;
#pragma unroll
    for (int m = 0; m < MAXCH; ++m) {
        const int i0 = (et + NROW * m) * 8;
        if (i0 >= d) continue;
        float sh[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        uint4 mu4[NMIX];
#pragma unroll
        for (int q = 0; q < NMIX; ++q)
            mu4[q] = *reinterpret_cast<const uint4 *>((NMIX == 6 ? p.mu[q] : p.fxk) + lo + i0);
        if (ok) ld8cg(shift + i0, sh);
#pragma unroll
        for (int q = 0; q < NMIX; ++q) {
            float mu[8], o[8];
            h8f(mu4[q], mu);
#pragma unroll
            for (int k = 0; k < 8; ++k) o[k] = v[m][k] + (sh[k] - v[m][k]) * mu[k];
            __half *dst = (NMIX == 6 ? p.xmix[q] : p.xk) + (size_t)b * d + i0;
            *reinterpret_cast<uint4 *>(dst) = fh8(o);
        }
        if (ok) st8(shift + i0, v[m]);
    }
}

// mode 0: time mix of layer l (layer 0 starts from the embedding + LN0),
// mode 1: channel mix of layer l, mode 2: final LayerNorm (head input).
// x[b] first receives the residual partial slabs of the preceding projection.
__device__ __forceinline__ void row_phase(const PkParams &p, SmemTail &t, int l, int b, int et, int mode) {
    const int d = p.d;
    const int slot = p.slots[b];
    const bool ok = slot >= 0 && slot < p.n_slots;
    float v[MAXCH][8];
    float *xr = p.x + (size_t)b * d;
    if (mode == 0 && l == 0) {
        int tok = p.tokens[b];
        if (et == 0) {
            if (!ok) atomicOr(p.err, ERR_SLOT);
            if (tok < 0 || tok >= p.V) atomicOr(p.err, ERR_TOKEN);
            if (ok) {
                const uint32_t bit = 1u << (slot & 31);
                if (atomicOr(p.dup + (slot >> 5), bit) & bit) atomicOr(p.err, ERR_DUP);
            }
        }
        if (tok < 0 || tok >= p.V) tok = 0;
#pragma unroll
        for (int m = 0; m < MAXCH; ++m) {
            const int i0 = (et + NROW * m) * 8;
#pragma unroll
            for (int k = 0; k < 8; ++k) v[m][k] = 0.0f;
            if (i0 < d) h8f(*reinterpret_cast<const uint4 *>(p.emb + (size_t)tok * d + i0), v[m]);
        }
        row_ln(v, d, et, p.ln0w, p.ln0b, t.red);
#pragma unroll
        for (int m = 0; m < MAXCH; ++m) {
            const int i0 = (et + NROW * m) * 8;
            if (i0 < d) st8(xr + i0, v[m]);
        }
    } else {
        const int ns = (mode == 1) ? p.s3 : p.s5;
#pragma unroll
        for (int m = 0; m < MAXCH; ++m) {
            const int i0 = (et + NROW * m) * 8;
#pragma unroll
            for (int k = 0; k < 8; ++k) v[m][k] = 0.0f;
            if (i0 < d) {
                // x and up to 8 slabs per batch, all loads issued before the adds
                const float *src = p.px + (size_t)b * d + i0;
                float4 xa = __ldcg(reinterpret_cast<const float4 *>(xr + i0));
                float4 xb = __ldcg(reinterpret_cast<const float4 *>(xr + i0 + 4));
                float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                for (int j0 = 0; j0 < ns; j0 += 8) {
                    float4 sa[8], sb[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        if (j0 + u < ns) {
                            const float *q = src + (size_t)(j0 + u) * p.xstride;
                            sa[u] = __ldcg(reinterpret_cast<const float4 *>(q));
                            sb[u] = __ldcg(reinterpret_cast<const float4 *>(q + 4));
                        } else {
                            sa[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                            sb[u] = sa[u];
                        }
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        acc[0] += sa[u].x; acc[1] += sa[u].y; acc[2] += sa[u].z; acc[3] += sa[u].w;
                        acc[4] += sb[u].x; acc[5] += sb[u].y; acc[6] += sb[u].z; acc[7] += sb[u].w;
                    }
                }
                v[m][0] = xa.x + acc[0]; v[m][1] = xa.y + acc[1]; v[m][2] = xa.z + acc[2]; v[m][3] = xa.w + acc[3];
                v[m][4] = xb.x + acc[4]; v[m][5] = xb.y + acc[5]; v[m][6] = xb.z + acc[6]; v[m][7] = xb.w + acc[7];
                if (mode != 2) st8(xr + i0, v[m]);
            }
        }
    }
    const size_t lo = (size_t)l * d;
    if (mode == 2) {
        row_ln(v, d, et, p.lnow, p.lnob, t.red);
#pragma unroll
        for (int m = 0; m < MAXCH; ++m) {
            const int i0 = (et + NROW * m) * 8;
            if (i0 < d) *reinterpret_cast<uint4 *>(p.xo + (size_t)b * d + i0) = fh8(v[m]);
        }
        return;
    }
    if (mode == 0)
        row_ln(v, d, et, p.ln1w + lo, p.ln1b + lo, t.red);
    else
        row_ln(v, d, et, p.ln2w + lo, p.ln2b + lo, t.red);
    float *shift = (mode == 0 ? p.shift_att : p.shift_ffn) + ((size_t)l * p.n_slots + (ok ? slot : 0)) * d;
    if (mode == 0)
        mix_out<6>(p, v, shift, ok, b, lo, et);
    else
        mix_out<1>(p, v, shift, ok, b, lo, et);
}

// Sum over the 64 row threads of one half (named barrier 2 + half).
__device__ __forceinline__ float half_sum(float v, float *red2, int hf, int et) {
    v = warp_sum(v);
    if ((et & 31) == 0) red2[2 * hf + ((et >> 5) & 1)] = v;
    named_bar(BAR_HALF + hf, 64);
    const float s = red2[2 * hf] + red2[2 * hf + 1];
    named_bar(BAR_HALF + hf, 64);
    return s;
}

// Inputs of one (slot, head) pair for channel j of the head, read from global
// memory one stage ahead of their use.  r, k, v are the sums of the projection's
// split-K slabs (slab order).
struct PairIn {
    float r, k, v, a, dec, g, vg, vf;
    float kk, ka, rk, lw, lb;
    int slot;
};
__device__ __forceinline__ void pair_load(const PkParams &p, int l, int pair, int j, PairIn &in) {
    const int b = pair / p.H, h = pair - (pair / p.H) * p.H;
    const size_t off = (size_t)b * p.d + (size_t)h * HS + j;
    const size_t wc = (size_t)l * p.d + (size_t)h * HS + j;
    in.slot = p.slots[b];
    float rr = 0.f, kk = 0.f, vv = 0.f;
#pragma unroll 4
    for (int s = 0; s < p.s1; ++s) {
        const size_t o = (size_t)s * p.xstride + off;
        rr += __ldcg(p.pr + o);
        kk += __ldcg(p.pk + o);
        vv += __ldcg(p.pv + o);
    }
    in.r = rr;
    in.k = kk;
    in.v = vv;
    in.a = __ldcg(p.a + off);
    in.dec = __ldcg(p.dec + off);
    in.g = __ldcg(p.gate + off);
    if (l > 0) {
        in.vg = __ldcg(p.vg + off);
        in.vf = __ldcg(p.vfirst + off);
    } else {
        in.vg = 0.f;
        in.vf = 0.f;
    }
    in.kk = __half2float(p.k_k[wc]);
    in.ka = __half2float(p.k_a[wc]);
    in.rk = __half2float(p.r_k[wc]);
    in.lw = __half2float(p.lnxw[wc]);
    in.lb = __half2float(p.lnxb[wc]);
}

// WKV7 of one (slot row b, head h) pair by the 64 threads of half `hf`; thread
// j owns state row j (value index j) of the 64x64 state at S in shared memory
// (row i = value index, column = key index) and channel j of the head's vectors:
//   kh = normalize(k * k_k), kp = k * (1 + (a - 1) * k_a),
//   vp = v (layer 0, also kept as v_first) or v + (v_first - v) * vg,
//   S[i][c] <- S[i][c] dec_c - (sum_m S[i][m] kh_m) kh_c a_c + vp_i kp_c,  y_i = sum_c S[i][c] r_c,
//   z_i = (GroupNorm(y)_i * gamma + beta + (sum_c r_c kp_c r_k_c) vp_i) * g_i  -> fp16.
// Row j is read in 16-byte chunks starting at chunk j (mod 16) so that the 8
// threads of a shared-memory phase hit 8 different bank groups.  The new state
// goes back to HBM with one bulk copy issued by the half's first thread.
__device__ __forceinline__ void wkv_pair(const PkParams &p, SmemTail &t, int l, int pair, const PairIn &in, float *S, int hf, int j,
                         int et) {
    const int b = pair / p.H, h = pair - (pair / p.H) * p.H;
    const bool ok = in.slot >= 0 && in.slot < p.n_slots;
    const size_t off = (size_t)b * p.d + (size_t)h * HS + j;
    float *red2 = t.red + 4;
    // per-channel vectors
    const float kk = in.k * in.kk;
    const float ss = half_sum(kk * kk, red2, hf, et);
    const float khv = kk / fmaxf(sqrtf(ss), 1e-12f);
    const float kpv = in.k * (1.0f + (in.a - 1.0f) * in.ka);
    float vpv;
    if (l == 0) {
        vpv = in.v;
        p.vfirst[off] = in.v;
    } else {
        vpv = in.v + (in.vf - in.v) * in.vg;
    }
    const float bonus = half_sum(in.r * kpv * in.rk, red2, hf, et);
    t.vkh[hf][j] = khv;
    t.vka[hf][j] = khv * in.a;
    t.vdec[hf][j] = in.dec;
    t.vkp[hf][j] = kpv;
    t.vr[hf][j] = in.r;
    named_bar(BAR_HALF + hf, 64);
    // row j of the state
    float4 row[16];
    float *Sr = S + j * HS;
    float sa = 0.0f;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
        const int cc = ((c + j) & 15) * 4;
        row[c] = ok ? *(const float4 *)(Sr + cc) : make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 kh = *(const float4 *)&t.vkh[hf][cc];
        sa += row[c].x * kh.x + row[c].y * kh.y + row[c].z * kh.z + row[c].w * kh.w;
    }
    float y = 0.0f;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
        const int cc = ((c + j) & 15) * 4;
        const float4 dc = *(const float4 *)&t.vdec[hf][cc];
        const float4 ka = *(const float4 *)&t.vka[hf][cc];
        const float4 kp = *(const float4 *)&t.vkp[hf][cc];
        const float4 rr = *(const float4 *)&t.vr[hf][cc];
        float4 sv = row[c];
        sv.x = sv.x * dc.x - sa * ka.x + vpv * kp.x;
        sv.y = sv.y * dc.y - sa * ka.y + vpv * kp.y;
        sv.z = sv.z * dc.z - sa * ka.z + vpv * kp.z;
        sv.w = sv.w * dc.w - sa * ka.w + vpv * kp.w;
        y += sv.x * rr.x + sv.y * rr.y + sv.z * rr.z + sv.w * rr.w;
        row[c] = sv;
    }
#pragma unroll
    for (int c = 0; c < 16; ++c) *(float4 *)(Sr + ((c + j) & 15) * 4) = row[c];
    fence_proxy_async();  // the bulk copy below reads what this thread wrote
    // GroupNorm over the head, bonus, gate
    const float mean = half_sum(y, red2, hf, et) * (1.0f / HS);
    const float dv = y - mean;
    const float var = half_sum(dv * dv, red2, hf, et) * (1.0f / HS);
    const float yn = dv * (1.0f / sqrtf(var + 64e-5f)) * in.lw + in.lb;
    p.z[off] = __float2half_rn((yn + bonus * vpv) * in.g);
    if (j == 0 && ok) {  // every row of this pair was written before the last half barrier
        float *dst = p.wkv + (((size_t)l * p.n_slots + in.slot) * p.H + h) * (HS * HS);
        bulk_s2g(dst, S, PAIR_B);
        bulk_commit();
    }
}

// ---------------------------------------------------------------------------
// Row-thread helpers that keep the 128 threads on one control path: thread 0
// waits, the outcome is broadcast through shared memory.
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool row_wait_count(const PkParams &p, SmemTail &t, const uint32_t *c, uint32_t target, int et) {
    if (et == 0) {
        *(volatile uint32_t *)(p.prog + 4 * blockIdx.x + 3) = 0x20000000u | (uint32_t)(c - p.cnt);
        const bool ok = wait_count(c, target, p.abort_flag);
        if (!ok) {
            if (!aborted(p.abort_flag)) note(p, 4u, (uint32_t)(c - p.cnt), ld_acquire(c), target, 0u);
            give_up(p);
        }
        t.flag = ok ? 1u : 0u;
    }
    named_bar(BAR_ROW, NROW);
    const bool ok = t.flag != 0u;
    named_bar(BAR_ROW, NROW);
    return ok;
}
__device__ __forceinline__ bool row_wait_mbar(const PkParams &p, SmemTail &t, uint64_t *bar, uint32_t parity, int et,
                              uint32_t what) {
    if (et == 0) {
        const bool ok = pk_mbar_wait(bar, parity, p.abort_flag);
        if (!ok) {
            if (!aborted(p.abort_flag)) note(p, 5u, what, parity, 0u, 0u);
            give_up(p);
        }
        t.flag = ok ? 1u : 0u;
    }
    named_bar(BAR_ROW, NROW);
    const bool ok = t.flag != 0u;
    named_bar(BAR_ROW, NROW);
    if (ok) (void)mbar_try_wait(bar, parity);  // completed phase: observe it from every thread
    return ok;
}

struct Ring {
    uint8_t *w, *x;
    uint64_t *full, *empty, *accf, *acce, *mma_done;
    uint32_t slot_w, slot_x, xkb;
    int ns;
};

// Epilogues of this CTA's items of one GEMM phase.
__device__ __forceinline__ bool row_gemm(const PkParams &p, SmemTail &t, const Ring &rg, uint32_t tmem, int l, int ph, int &nacc,
                         int c, int G, int et) {
    const PkGemm &g = t.g[gemm_of(l, ph)];
    uint32_t *done = (ph == PH_HEAD) ? p.cnt + p.L * PK_NPH + 1 : p.cnt + l * PK_NPH + ph;
    const int warp = (et >> 5) + 2, lane = et & 31, qd = warp & 3;
    for (int i = first_of(c, G, g.nitems), e = first_of(c + 1, G, g.nitems); i < e; ++i) {
        const PItem it = locate(g, i, p.kbs);
        const PkSeg sg = g.seg[it.s];  // register copy: the stores below cannot alias it
        const int buf = nacc & 1;
        if (et == 0)
            *(volatile uint32_t *)(p.prog + 4 * c + 3) = 0x80000000u | ((uint32_t)l << 16) | ((uint32_t)ph << 12) | (uint32_t)nacc;
        if (!row_wait_mbar(p, t, &rg.accf[buf], (uint32_t)(nacc >> 1) & 1u, et,
                           0x10000000u | ((uint32_t)l << 16) | ((uint32_t)ph << 12) | (uint32_t)nacc))
            return false;
        tc_fence_after();
        const uint32_t taddr = tmem + ((uint32_t)(qd * 32) << 16) + (uint32_t)(buf * p.npad);
        const int n = it.tile * GEMM_TILE_M + qd * 32 + lane;
        const bool valid = it.kb1 > it.kb0;
        float bias = 0.0f;
        if ((sg.epi == EPI_DECAY || sg.epi == EPI_SIGMOID_BIAS) && n < sg.rows)
            bias = __half2float(sg.bias[(size_t)l * sg.bias_stride + n]);
        const bool split_fix = sg.fix && sg.S > 1;
        if (sg.fix && sg.S == 1)
            epi_final(sg, false, taddr, valid, n, p.npad, p.B, bias);
        else
            epi_partial(sg, taddr, valid, n, it.split, p.npad, p.B);
        tc_fence_before();
        mbar_arrive(&rg.acce[buf]);
        ++nacc;
        if (split_fix) {
            named_bar(BAR_ROW, NROW);
            if (et == 0) {
                __threadfence();
                uint32_t *tc = p.tcnt + (size_t)l * p.tcnt_layer + sg.cnt0 + it.tile;
                const uint32_t old = atomicAdd(tc, 1u);
                __threadfence();
                t.flag = (old == (uint32_t)(sg.S - 1)) ? 1u : 0u;
            }
            named_bar(BAR_ROW, NROW);
            if (t.flag) epi_final(sg, true, 0u, true, n, p.npad, p.B, bias);
        }
    }
    const int mine = first_of(c + 1, G, g.nitems) - first_of(c, G, g.nitems);
    named_bar(BAR_ROW, NROW);  // every output of this CTA's items is stored
    if (et == 0 && mine > 0) signal_count(done, (uint32_t)mine);
    return true;
}

__device__ __forceinline__ void row_role(const PkParams &p, SmemTail &t, const Ring &rg, uint32_t tmem, int c, int G, int et) {
    int q = 0, nacc = 0;
    uint32_t nstate = 0;
    const int r0 = first_of(c, G, p.B), r1 = first_of(c + 1, G, p.B);
    const int npairs = p.B * p.H;
    for (int l = 0; l < p.L; ++l) {
        uint32_t *cnt = p.cnt + l * PK_NPH;
        // LN1 + time-mix shifts
        if (l > 0 && !row_wait_count(p, t, cnt - PK_NPH + PH_G5, (uint32_t)t.g[PKG_G5].nitems, et)) return;
        for (int b = r0; b < r1; ++b) row_phase(p, t, l, b, et, 0);
        named_bar(BAR_ROW, NROW);
        if (et == 0 && r1 > r0) signal_count(cnt + PH_LN1, (uint32_t)(r1 - r0));
        // r, k, v + LoRA-down; LoRA-up
        if (!row_gemm(p, t, rg, tmem, l, PH_G1, nacc, c, G, et)) return;
        q += gemm_stages(t.g[gemm_of(l, PH_G1)], c, G, p.kbs);
        if (!row_gemm(p, t, rg, tmem, l, PH_G2, nacc, c, G, et)) return;
        q += gemm_stages(t.g[gemm_of(l, PH_G2)], c, G, p.kbs);
        // WKV over this CTA's (slot, head) pairs, states from the ring; half hf of
        // the row threads takes pair ps + hf of each stage, inputs loaded a stage ahead
        if (!row_wait_count(p, t, cnt + PH_G2, (uint32_t)t.g[gemm_of(l, PH_G2)].nitems, et)) return;
        {
            const int hf = et >> 6, j = et & 63;
            const int p0 = first_of(c, G, npairs), pe = first_of(c + 1, G, npairs);
            PairIn cur, nxt;
            if (p0 + hf < pe && hf < p.kbs) pair_load(p, l, p0 + hf, j, cur);
            for (int ps = p0; ps < pe; ps += p.kbs) {
                const int slot = q % rg.ns;
                const int mine = ps + hf;
                const bool act = hf < p.kbs && mine < pe;
                const bool more = hf < p.kbs && mine + p.kbs < pe;
                if (more) pair_load(p, l, mine + p.kbs, j, nxt);
                if (et == 0) *(volatile uint32_t *)(p.prog + 4 * c + 3) = 0x40000000u | ((uint32_t)l << 16) | (uint32_t)q;
                if (!row_wait_mbar(p, t, &rg.full[slot], (uint32_t)(q / rg.ns) & 1u, et,
                                   0x20000000u | ((uint32_t)l << 16) | (uint32_t)q))
                    return;
                if (act) wkv_pair(p, t, l, mine, cur, (float *)(rg.w + (size_t)slot * rg.slot_w + (size_t)hf * PAIR_B), hf, j, et);
                if (et == 64 && act) bulk_wait_read_all();  // the second half's copy has read its part of the slot
                named_bar(BAR_ROW, NROW);
                ++nstate;
                if (et == 0) {
                    bulk_wait_read_all();
                    mbar_arrive(&rg.empty[slot]);
                    *(volatile uint32_t *)&t.state_done = nstate;
                }
                if (more) cur = nxt;
                ++q;
            }
            named_bar(BAR_ROW, NROW);  // every z of this CTA's pairs is stored
            if (et == 0 && pe > p0) signal_count(cnt + PH_WKV, (uint32_t)(pe - p0));
        }
        // output projection; LN2 + channel-mix shift; key; value
        if (!row_gemm(p, t, rg, tmem, l, PH_G3, nacc, c, G, et)) return;
        q += gemm_stages(t.g[PKG_G3], c, G, p.kbs);
        if (!row_wait_count(p, t, cnt + PH_G3, (uint32_t)t.g[PKG_G3].nitems, et)) return;
        for (int b = r0; b < r1; ++b) row_phase(p, t, l, b, et, 1);
        named_bar(BAR_ROW, NROW);
        if (et == 0 && r1 > r0) signal_count(cnt + PH_LN2, (uint32_t)(r1 - r0));
        if (!row_gemm(p, t, rg, tmem, l, PH_G4, nacc, c, G, et)) return;
        q += gemm_stages(t.g[PKG_G4], c, G, p.kbs);
        if (!row_gemm(p, t, rg, tmem, l, PH_G5, nacc, c, G, et)) return;
        q += gemm_stages(t.g[PKG_G5], c, G, p.kbs);
    }
    if (!p.head) return;
    if (!row_wait_count(p, t, p.cnt + (p.L - 1) * PK_NPH + PH_G5, (uint32_t)t.g[PKG_G5].nitems, et)) return;
    for (int b = r0; b < r1; ++b) row_phase(p, t, p.L, b, et, 2);
    named_bar(BAR_ROW, NROW);
    if (et == 0 && r1 > r0) signal_count(p.cnt + p.L * PK_NPH, (uint32_t)(r1 - r0));
    row_gemm(p, t, rg, tmem, p.L, PH_HEAD, nacc, c, G, et);
}

// ---------------------------------------------------------------------------
// MMA issuer (one thread).
// ---------------------------------------------------------------------------
// The ring's slots are shared by the MMA's stages and the row threads' state
// stages; the MMA skips the latter.  Before it waits on a slot's `full`
// barrier by phase parity, every earlier state stage must have been released,
// or the barrier could still be in a phase two uses behind and the parity test
// would pass on the wrong phase.
__device__ bool mma_wait_states(const PkParams &p, const SmemTail &t, uint32_t need) {
    if (*(volatile const uint32_t *)&t.state_done >= need) return true;
    const uint64_t t0 = gtimer();
    for (uint32_t it = 1;; ++it) {
        if (*(volatile const uint32_t *)&t.state_done >= need) return true;
        __nanosleep(128);
        if ((it & 63u) == 0) {
            if (aborted(p.abort_flag)) return false;
            if (gtimer() - t0 > WAIT_LIMIT_NS) return false;
        }
    }
}

__device__ void mma_gemm(const PkParams &p, const SmemTail &t, const Ring &rg, uint32_t tmem, uint32_t idesc, int l,
                         int ph, int &q, int &nacc, int c, int G, bool &ok, uint32_t need_state) {
    if (need_state && !mma_wait_states(p, t, need_state)) {
        if (!aborted(p.abort_flag)) note(p, 6u, need_state, (uint32_t)q, ((uint32_t)l << 8) | (uint32_t)ph, 0u);
        ok = false;
        return;
    }
    const PkGemm &g = t.g[gemm_of(l, ph)];
    for (int i = first_of(c, G, g.nitems), e = first_of(c + 1, G, g.nitems); i < e && ok; ++i) {
        const PItem it = locate(g, i, p.kbs);
        const int buf = nacc & 1;
        if (nacc >= 2 && !pk_mbar_wait(&rg.acce[buf], (uint32_t)((nacc >> 1) - 1) & 1u, p.abort_flag)) {
            if (!aborted(p.abort_flag)) note(p, 2u, (uint32_t)nacc, (uint32_t)q, ((uint32_t)l << 8) | (uint32_t)ph, 0u);
            ok = false;
            break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(buf * p.npad);
        uint32_t issued = 0;
        for (int kb = it.kb0; kb < it.kb1; kb += p.kbs) {
            const int slot = q % rg.ns;
            *(volatile uint32_t *)(p.prog + 4 * c + 2) = (uint32_t)q | ((uint32_t)nacc << 16);
            if (!pk_mbar_wait(&rg.full[slot], (uint32_t)(q / rg.ns) & 1u, p.abort_flag)) {
                if (!aborted(p.abort_flag))
                    note(p, 3u, (uint32_t)q, (uint32_t)nacc, ((uint32_t)l << 8) | (uint32_t)ph, (uint32_t)kb);
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t a0 = smem_u32(rg.w + (size_t)slot * rg.slot_w);
            const uint32_t b0 = smem_u32(rg.x + (size_t)slot * rg.slot_x);
            for (int kk = 0; kk < p.kbs * (GEMM_TILE_K / 16); ++kk)
                mma_f16(d_tmem, sdesc_k128(a0 + (kk >> 2) * TILE_B + (kk & 3) * 32),
                        sdesc_k128(b0 + (kk >> 2) * rg.xkb + (kk & 3) * 32), idesc, (issued | (uint32_t)kk) ? 1u : 0u);
            issued = 1;
            mma_commit(&rg.empty[slot]);
            ++q;
        }
        if (!ok) break;
        if (issued)
            mma_commit(&rg.accf[buf]);
        else
            mbar_arrive(&rg.accf[buf]);
        ++nacc;
    }
}

__device__ void mma_role(const PkParams &p, const SmemTail &t, const Ring &rg, uint32_t tmem, int c, int G) {
    const uint32_t idesc = idesc_f16(GEMM_TILE_M, p.npad);
    int q = 0, nacc = 0;
    bool ok = true;
    const int npairs = p.B * p.H;
    const uint32_t ws = (uint32_t)wkv_stages(c, G, npairs, p.kbs);
    uint32_t need = 0;  // state stages skipped so far
    for (int l = 0; l < p.L && ok; ++l) {
        mma_gemm(p, t, rg, tmem, idesc, l, PH_G1, q, nacc, c, G, ok, need);
        if (ok) mma_gemm(p, t, rg, tmem, idesc, l, PH_G2, q, nacc, c, G, ok, need);
        q += (int)ws;
        need += ws;
        if (ok) mma_gemm(p, t, rg, tmem, idesc, l, PH_G3, q, nacc, c, G, ok, need);
        if (ok) mma_gemm(p, t, rg, tmem, idesc, l, PH_G4, q, nacc, c, G, ok, need);
        if (ok) mma_gemm(p, t, rg, tmem, idesc, l, PH_G5, q, nacc, c, G, ok, need);
    }
    if (ok && p.head) mma_gemm(p, t, rg, tmem, idesc, p.L, PH_HEAD, q, nacc, c, G, ok, need);
    if (!ok) give_up(p);
    // every MMA issued here has finished before the accumulators are freed
    mma_commit(rg.mma_done);
    const uint64_t t0 = gtimer();
    while (!mbar_try_wait(rg.mma_done, 0u) && gtimer() - t0 < WAIT_LIMIT_NS) {
    }
}

// ---------------------------------------------------------------------------
// Producer (one thread): weight tiles and states in ring order; activation
// boxes of a stage once its producing phase is complete.
// ---------------------------------------------------------------------------
__device__ void producer_role(const PkParams &p, const SmemTail &t, const Ring &rg, int c, int G) {
    const uint64_t polW = policy_evict_first(), polX = policy_evict_last();
    Cursor wc, xc;
    cur_begin(wc, p, t, c, G);
    cur_begin(xc, p, t, c, G);
    int qw = 0, qx = 0;
    int xl = -1, xph = -1;
    bool xready = false;
    uint64_t t_idle = 0;
    uint32_t spins = 0;
    bool ok = true;
    while (!xc.done) {
        bool prog = false;
        if (qx < qw) {
            if (xc.ph == PH_WKV) {
                cur_next(xc, p, t, c, G);
                ++qx;
                prog = true;
            } else {
                if (xc.l != xl || xc.ph != xph) {
                    xl = xc.l;
                    xph = xc.ph;
                    xready = false;
                }
                if (!xready) {
                    const uint32_t *dc;
                    uint32_t tg;
                    x_dep(p, t, xl, xph, &dc, &tg);
                    xready = ld_acquire(dc) >= tg;
                    if (xready) fence_proxy_async_global();
                }
                if (xready) {
                    const PkSeg &sg = t.g[gemm_of(xc.l, xc.ph)].seg[xc.s];
                    const int slot = qx % rg.ns;
                    mbar_expect_tx(&rg.full[slot], (uint32_t)p.kbs * rg.xkb);
                    if (sg.x3) {
                        tma_load_3d(rg.x + (size_t)slot * rg.slot_x, &p.maps[sg.xmap], &rg.full[slot], 0, 0, xc.kb, polX);
                    } else {
                        for (int h = 0; h < p.kbs; ++h)
                            tma_load_2d(rg.x + (size_t)slot * rg.slot_x + (size_t)h * rg.xkb, &p.maps[sg.xmap],
                                        &rg.full[slot], (xc.kb + h) * GEMM_TILE_K, 0, polX);
                    }
                    cur_next(xc, p, t, c, G);
                    ++qx;
                    prog = true;
                }
            }
        }
        if (!wc.done && (qw < rg.ns || mbar_try_wait(&rg.empty[qw % rg.ns], (uint32_t)((qw / rg.ns) - 1) & 1u))) {
            const int slot = qw % rg.ns;
            uint8_t *dst = rg.w + (size_t)slot * rg.slot_w;
            if (wc.ph == PH_WKV) {
                const int np = min(p.kbs, wc.iend - wc.i);
                mbar_expect_tx(&rg.full[slot], (uint32_t)np * PAIR_B);
                for (int k = 0; k < np; ++k) {
                    const int pair = wc.i + k;
                    const int b = pair / p.H, h = pair - (pair / p.H) * p.H;
                    int sl = p.slots[b];
                    if (sl < 0 || sl >= p.n_slots) sl = 0;
                    const float *src = p.wkv + (((size_t)wc.l * p.n_slots + sl) * p.H + h) * (HS * HS);
                    bulk_g2s(dst + (size_t)k * PAIR_B, src, PAIR_B, &rg.full[slot]);
                }
            } else {
                const PkSeg &sg = t.g[gemm_of(wc.l, wc.ph)].seg[wc.s];
                mbar_expect_tx_noarrive(&rg.full[slot], rg.slot_w);
                const int tb = sg.layer_tiles * (wc.ph == PH_HEAD ? 0 : wc.l) + wc.tile * sg.kb + wc.kb;
                tma_load_3d(dst, &p.maps[sg.wmap], &rg.full[slot], 0, 0, tb, polW);
            }
            cur_next(wc, p, t, c, G);
            ++qw;
            prog = true;
        }
        if (prog) {
            spins = 0;
            t_idle = 0;
            *(volatile uint32_t *)(p.prog + 4 * c) = (uint32_t)qw;
            *(volatile uint32_t *)(p.prog + 4 * c + 1) = (uint32_t)qx | (xready ? 0x80000000u : 0u) |
                                                         ((uint32_t)xc.ph << 24) | ((uint32_t)xc.l << 16);
        } else if (++spins > 2 && (__nanosleep(32), (spins & 63u) == 0)) {
            const uint64_t now = gtimer();
            if (t_idle == 0) {
                t_idle = now;
            } else if (now - t_idle > WAIT_LIMIT_NS || aborted(p.abort_flag)) {
                if (!aborted(p.abort_flag))
                    note(p, 1u, (uint32_t)qw, (uint32_t)qx, ((uint32_t)xc.l << 8) | (uint32_t)xc.ph,
                         ((uint32_t)wc.l << 8) | (uint32_t)wc.ph | (xready ? 0x10000u : 0u) | (wc.done ? 0x20000u : 0u));
                ok = false;
                break;
            }
        }
    }
    if (!ok) {
        give_up(p);
        // wait (bounded) for the copies still in flight into this CTA's ring
        const uint64_t t0 = gtimer();
        for (int j = (qw > rg.ns ? qw - rg.ns : 0); j < qw; ++j)
            while (!mbar_try_wait(&rg.full[j % rg.ns], (uint32_t)(j / rg.ns) & 1u) && gtimer() - t0 < WAIT_LIMIT_NS) {
            }
    }
}

__global__ void __launch_bounds__(PK_THREADS, 1) decode_persistent_kernel(const __grid_constant__ PkParams p) {
    extern __shared__ uint8_t smem_raw[];
    // offsets from the shared array itself keep the compiler aware that every
    // pointer below addresses shared memory
    uint8_t *base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    Ring rg;
    rg.ns = p.stages;
    rg.xkb = (uint32_t)p.npad * 128u;
    rg.slot_w = (uint32_t)p.kbs * TILE_B;
    rg.slot_x = (uint32_t)p.kbs * rg.xkb;
    rg.w = base;
    rg.x = base + (size_t)rg.ns * rg.slot_w;
    rg.full = (uint64_t *)(rg.x + (size_t)rg.ns * rg.slot_x);
    rg.empty = rg.full + rg.ns;
    rg.accf = rg.empty + rg.ns;
    rg.acce = rg.accf + 2;
    rg.mma_done = rg.acce + 2;
    uint8_t *tail = reinterpret_cast<uint8_t *>(rg.mma_done + 1);
    tail += (16u - (smem_u32(tail) & 15u)) & 15u;
    SmemTail &t = *reinterpret_cast<SmemTail *>(tail);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x, G = gridDim.x;

    {  // phase tables into shared memory
        const uint32_t *src = (const uint32_t *)&p.g[0];
        uint32_t *dst = (uint32_t *)&t.g[0];
        for (int i = threadIdx.x; i < (int)(sizeof(PkGemm) * PKG_COUNT / 4); i += PK_THREADS) dst[i] = src[i];
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < rg.ns; ++i) {
            mbar_init(&rg.full[i], 1);
            mbar_init(&rg.empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&rg.accf[i], 1);
            mbar_init(&rg.acce[i], NROW);
        }
        mbar_init(rg.mma_done, 1);
        t.state_done = 0u;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0)
        for (int i = 0; i < p.nmaps; ++i) prefetch_tmap(&p.maps[i]);
    __syncthreads();
    if (warp == 1) {
        tmem_alloc(&t.tmem_base, (uint32_t)p.ncols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = t.tmem_base;

    if (warp == 0) {
        if (lane == 0) producer_role(p, t, rg, c, G);
    } else if (warp == 1) {
        if (lane == 0) mma_role(p, t, rg, tmem, c, G);
    } else {
        row_role(p, t, rg, tmem, c, G, threadIdx.x - 64);
        if (threadIdx.x == 64) bulk_wait_all();  // state write-backs complete before exit
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, (uint32_t)p.ncols);
    }
}

}  // namespace

size_t pk_smem_bytes(int npad, int kbs, int stages) {
    const size_t slot = (size_t)kbs * TILE_B + (size_t)kbs * npad * 128;
    return 1024 + (size_t)stages * slot + (size_t)(2 * stages + 5) * 8 + 16 + sizeof(SmemTail);
}
int pk_max_stages(int npad, int kbs) {
    const size_t slot = (size_t)kbs * TILE_B + (size_t)kbs * npad * 128;
    const size_t fixed = 1024 + 5 * 8 + 16 + sizeof(SmemTail);
    const size_t budget = 227 * 1024 - fixed;
    int s = (int)(budget / (slot + 16));
    return s > 8 ? 8 : s;
}

void launch_persistent(const PkParams &p, int grid, size_t smem, cudaStream_t st, cudaError_t *e) {
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t r = cudaFuncSetAttribute(decode_persistent_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             227 * 1024);
        if (r != cudaSuccess) {
            *e = r;
            return;
        }
        attr_set = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(PK_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeCooperative;
    at[0].val.cooperative = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    cudaError_t r = cudaLaunchKernelEx(&cfg, decode_persistent_kernel, p);
    if (r != cudaSuccess) *e = r;
}

}  // namespace rk
