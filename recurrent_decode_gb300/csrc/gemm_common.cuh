// gemm_common.cuh -- pieces shared by the fp16 and int8-weight tensor-core GEMM
// kernels (gemm.cu, gemm8.cu): tile constants, the per-kind epilogue from tensor
// memory, and the work partition into (row tile, k-split) items.
#pragma once
#include "internal.cuh"

namespace rk {

constexpr uint32_t W_TILE_BYTES = GEMM_TILE_M * GEMM_TILE_K * 2;  // 16 KB
// A pipeline stage holds KB_STAGE consecutive k-blocks: one TMA copy of the
// adjacent weight tiles (32 KB) and one activation box per k-block.
constexpr int KB_STAGE = 2;
constexpr uint32_t W_STAGE_BYTES = KB_STAGE * W_TILE_BYTES;


// Apply the segment's epilogue to one result.  Returns true when EPI_RELU2
// stores a nonzero fp16 value (so the caller can record sparsity).
__device__ __forceinline__ bool epi_store(const GemmSeg &s, int n, int b, float acc, float bias) {
    size_t o = (size_t)b * s.ldo + n;
    switch (s.epi) {
        case EPI_F32: ((float *)s.out)[o] = acc; break;
        case EPI_F16: ((__half *)s.out)[o] = __float2half_rn(acc); break;
        case EPI_F16_TANH: ((__half *)s.out)[o] = __float2half_rn(fast_tanh(acc)); break;
        case EPI_F16_SIGMOID: ((__half *)s.out)[o] = __float2half_rn(fast_sigmoid(acc)); break;
        case EPI_DECAY: ((float *)s.out)[o] = rwkv_decay(bias + acc); break;
        case EPI_SIGMOID_BIAS: ((float *)s.out)[o] = fast_sigmoid(bias + acc); break;
        case EPI_RESID: ((float *)s.out)[o] += acc; break;
        case EPI_RELU2: {
            float t = fmaxf(acc, 0.0f);
            __half h = __float2half_rn(t * t);
            ((__half *)s.out)[o] = h;
            return __half2float(h) != 0.0f;
        }
        default: break;
    }
    return false;
}

// Epilogue warps: EPI_GROUPS per TMEM lane quarter (a warp may only read its
// own quarter's 32 lanes); group g of a quarter takes the column chunks
// g, g + EPI_GROUPS, ... of EPI_CW slot columns each, so that a wide batch's
// epilogue is spread over many warps instead of running as one latency chain
// per sub-partition.
constexpr int EPI_GROUPS = 4;
constexpr int EPI_WARPS = 4 * EPI_GROUPS;
constexpr int EPI_THREADS = EPI_WARPS * 32;
constexpr int EPI_CW = 16;
constexpr int GEMM_TC_THREADS = 64 + EPI_THREADS;

// One chunk of accumulator columns into registers (a 32-column chunk may be the
// 16-column tail of the accumulator: the rest reads as zero).
__device__ __forceinline__ void chunk_ld(uint32_t taddr, float (&v)[16], bool) { tmem_ld16(taddr, v); }
__device__ __forceinline__ void chunk_ld(uint32_t taddr, float (&v)[32], bool full) {
    if (full) {
        tmem_ld32(taddr, v);
    } else {
        float h[16];
        tmem_ld16(taddr, h);
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            v[q] = h[q];
            v[q + 16] = 0.0f;
        }
    }
}

// Epilogue of one finished accumulator (one weight row n per thread, npad slot
// columns in TMEM; npad is a multiple of 16): the kind is dispatched once, then
// a straight-line loop per chunk of EPI_CW columns starting at column c0.
// Split items store raw fp32 partials (slab `split`).  Every lane executes the
// TMEM loads (they are warp-collective); stores are guarded.
template <int KIND>
__device__ __forceinline__ bool epi_run(const GemmSeg &sg, uint32_t taddr, bool valid, int n, int split, int npad,
                                        int B, int c0, float bias) {
    const bool live = n < sg.rows;
    const bool scaled = sg.wscale != nullptr;  // int8 weights: the row sum times the row's scale
    const float wsc = scaled && live ? __half2float(sg.wscale[n]) : 1.0f;
    bool nz = false;
    for (int cb = c0; cb < npad; cb += EPI_GROUPS * EPI_CW) {
        float v[EPI_CW];
        if (valid) {
            chunk_ld(taddr + (uint32_t)cb, v, cb + EPI_CW <= npad);
        } else {
#pragma unroll
            for (int q = 0; q < EPI_CW; ++q) v[q] = 0.0f;
        }
        if (!live) continue;
        if (scaled) {
#pragma unroll
            for (int q = 0; q < EPI_CW; ++q) v[q] *= wsc;
        }
        const int nq = min(EPI_CW, B - cb);
        if (KIND == -1) {  // raw fp32 partial
            float *out = (float *)sg.out + (size_t)split * sg.split_stride + (size_t)cb * sg.ldo + n;
#pragma unroll
            for (int q = 0; q < EPI_CW; ++q)
                if (q < nq) out[(size_t)q * sg.ldo] = v[q];
        } else if (KIND == EPI_RESID) {
            float *out = (float *)sg.out + (size_t)cb * sg.ldo + n;
            float old[EPI_CW];
#pragma unroll
            for (int q = 0; q < EPI_CW; ++q) old[q] = q < nq ? out[(size_t)q * sg.ldo] : 0.0f;
#pragma unroll
            for (int q = 0; q < EPI_CW; ++q)
                if (q < nq) out[(size_t)q * sg.ldo] = old[q] + v[q];
        } else if (KIND == EPI_F32 || KIND == EPI_DECAY || KIND == EPI_SIGMOID_BIAS) {
            float *out = (float *)sg.out + (size_t)cb * sg.ldo + n;
#pragma unroll
            for (int q = 0; q < EPI_CW; ++q) {
                float y = v[q];
                if (KIND == EPI_DECAY) y = rwkv_decay(bias + y);
                if (KIND == EPI_SIGMOID_BIAS) y = fast_sigmoid(bias + y);
                if (q < nq) out[(size_t)q * sg.ldo] = y;
            }
        } else {  // fp16 outputs
            __half *out = (__half *)sg.out + (size_t)cb * sg.ldo + n;
#pragma unroll
            for (int q = 0; q < EPI_CW; ++q) {
                float y = v[q];
                if (KIND == EPI_F16_TANH) y = fast_tanh(y);
                if (KIND == EPI_F16_SIGMOID) y = fast_sigmoid(y);
                if (KIND == EPI_RELU2) {
                    y = fmaxf(y, 0.0f);
                    y = y * y;
                }
                const __half hy = __float2half_rn(y);
                if (q < nq) {
                    out[(size_t)q * sg.ldo] = hy;
                    if (KIND == EPI_RELU2) nz |= __half2float(hy) != 0.0f;
                }
            }
        }
    }
    return nz;
}

// Out of line: one copy of the epilogue code serves every item.  Inlined at
// each call site the kernel's code grew past what the instruction cache keeps
// warm between items, and the graph-replayed step ran 2-4 % slower.
// `bias`: the segment's bias of row n (EPI_DECAY / EPI_SIGMOID_BIAS), loaded
// by the caller before it waits for the accumulator (see epi_bias).
static __device__ __noinline__ bool epi_item(const GemmSeg &sg, uint32_t taddr, bool valid, int n, int split,
                                             int npad, int B, int c0, float bias) {
    if (sg.S > 1) return epi_run<-1>(sg, taddr, valid, n, split, npad, B, c0, bias);
    switch (sg.epi) {
        case EPI_F32: return epi_run<EPI_F32>(sg, taddr, valid, n, split, npad, B, c0, bias);
        case EPI_F16: return epi_run<EPI_F16>(sg, taddr, valid, n, split, npad, B, c0, bias);
        case EPI_F16_TANH: return epi_run<EPI_F16_TANH>(sg, taddr, valid, n, split, npad, B, c0, bias);
        case EPI_F16_SIGMOID: return epi_run<EPI_F16_SIGMOID>(sg, taddr, valid, n, split, npad, B, c0, bias);
        case EPI_DECAY: return epi_run<EPI_DECAY>(sg, taddr, valid, n, split, npad, B, c0, bias);
        case EPI_SIGMOID_BIAS: return epi_run<EPI_SIGMOID_BIAS>(sg, taddr, valid, n, split, npad, B, c0, bias);
        case EPI_RESID: return epi_run<EPI_RESID>(sg, taddr, valid, n, split, npad, B, c0, bias);
        case EPI_RELU2: return epi_run<EPI_RELU2>(sg, taddr, valid, n, split, npad, B, c0, bias);
        default: return false;
    }
}
// Finish row n of a split tile (GemmSeg::fix_out): add the S partial slabs in
// slab order to zero, apply the fp16 kind fix_epi, store (the same arithmetic
// as the LoRA finalize kernel, so either path gives the same bits).  The slabs were written by
// other SMs: read through L2, the loads of up to FIX_BATCH slabs in flight at
// once (an L2 round trip under the weight stream costs about a microsecond).
// Columns as in epi_run.
constexpr int FIX_BATCH = 4;
__device__ __forceinline__ void fix_item(const GemmSeg &sg, int n, int npad, int B, int c0) {
    if (n >= sg.rows) return;
    constexpr int HW = EPI_CW / 2;  // columns per pass
    const int kind = sg.fix_epi;
    const float *src = (const float *)sg.out + n;
    __half *dst = (__half *)sg.fix_out + n;
    for (int cb = c0; cb < npad; cb += EPI_GROUPS * EPI_CW) {
        for (int h = cb; h < cb + EPI_CW; h += HW) {
            const int nq = min(HW, B - h);
            if (nq <= 0) break;
            float v[HW];
            for (int j0 = 0; j0 < sg.S; j0 += FIX_BATCH) {
                float t[FIX_BATCH][HW];
#pragma unroll
                for (int j = 0; j < FIX_BATCH; ++j) {
                    const float *sj = src + (size_t)(j0 + j) * sg.split_stride + (size_t)h * sg.ldo;
#pragma unroll
                    for (int q = 0; q < HW; ++q)
                        t[j][q] = (j0 + j < sg.S && q < nq) ? __ldcg(sj + (size_t)q * sg.ldo) : 0.0f;
                }
#pragma unroll
                for (int j = 0; j < FIX_BATCH; ++j)
#pragma unroll
                    for (int q = 0; q < HW; ++q)
                        if (j0 + j < sg.S) v[q] = ((j0 + j == 0) ? 0.0f : v[q]) + t[j][q];
            }
#pragma unroll
            for (int q = 0; q < HW; ++q) {
                float y = v[q];
                if (kind == EPI_F16_TANH) y = fast_tanh(y);
                else if (kind == EPI_F16_SIGMOID) y = fast_sigmoid(y);
                if (q < nq) dst[(size_t)(h + q) * sg.ldo] = __float2half_rn(y);
            }
        }
    }
}

// The bias an epilogue of weight row n needs (0 for kinds without one).
__device__ __forceinline__ float epi_bias(const GemmSeg &sg, int n) {
    return (sg.S == 1 && (sg.epi == EPI_DECAY || sg.epi == EPI_SIGMOID_BIAS) && n < sg.rows) ? __half2float(sg.bias[n])
                                                                                               : 0.0f;
}

// ---------------------------------------------------------------------------
// Work partition: global items numbered segment by segment, item = (row tile,
// split); CTA c owns items [first(c), first(c+1)).
// ---------------------------------------------------------------------------
__device__ __forceinline__ int item_first(int c, int G, int I) { return (int)(((long long)c * I) / G); }

struct Item {
    int s, tile, split, kb0, kb1;
};
__device__ __forceinline__ Item locate_item(const GemmSeg *seg, int nseg, int i) {
    int s = 0;
    while (s + 1 < nseg && i >= seg[s + 1].item0) ++s;
    const GemmSeg &g = seg[s];
    const int local = i - g.item0;
    Item it;
    it.s = s;
    it.tile = local / g.S;
    it.split = local - it.tile * g.S;
    const int np = g.kb / KB_STAGE;  // k-block pairs of the segment
    it.kb0 = (int)(((long long)it.split * np) / g.S) * KB_STAGE;
    it.kb1 = (int)(((long long)(it.split + 1) * np) / g.S) * KB_STAGE;
    return it;
}
// Flags of all-zero activation k-blocks, staged in shared memory (nullptr: none
// skipped).  A stage (k-blocks kb, kb+1) is skipped when both are all zero.
__device__ __forceinline__ bool kblock_skipped(const uint32_t *flags, int kblk) {
    return flags != nullptr && flags[kblk] == 0u;
}
__device__ __forceinline__ bool stage_skipped(const uint32_t *flags, int kb) {
    return flags != nullptr && flags[kb] == 0u && flags[kb + 1] == 0u;
}
constexpr int MAX_NZ_BLOCKS = 1024;  // d_ffn / 64


}  // namespace rk
