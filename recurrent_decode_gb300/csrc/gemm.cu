// gemm.cu -- skinny projection GEMMs of the decode step: Y[b][n] = sum_k X[b][k] W[n][k]
// for B slot rows (the activations) against fp16 weight matrices streamed once.
//
// The pages' decode kernels for this step are M=1 / split-K GEMVs written for
// consumer cards ("RWKV 批量推理中 Prefill 的正确打开方式", §三:
// linear_orig_row1_exact_f16_kernel, linear_f16_m1_splitk).  On sm_103a the
// same weight stream is fed to the 5th-generation tensor cores with the roles
// swapped: 128 weight rows form the MMA's M side, the B slots its N side (padded
// to 16), so one pass over the weights serves the whole batch.
//
//  * tensor-core kernel: one CTA per SM, warp-specialised -- warp 0 issues TMA
//    loads of 128x64 weight tiles and Bx64 activation tiles into a ring of
//    shared-memory stages, warp 1 issues tcgen05.mma into a TMEM accumulator,
//    warps 2-5 drain TMEM and apply the epilogue.  The (tile, k-block) units of
//    all segments are split evenly over the grid (stream-K); a tile whose
//    k-range spans several CTAs is reduced by the last CTA to arrive, summing
//    the partials in CTA order so the result does not depend on timing.
//  * SIMT kernel: a plain warp-per-row dot product with the same epilogues,
//    kept as an independent cross-check of the tensor-core kernel.
#include "internal.cuh"

namespace rk {

__device__ __forceinline__ float sigm(float x) { return 1.0f / (1.0f + expf(-x)); }

// Apply the segment's epilogue to one result.  Returns the fp16 value stored
// for EPI_RELU2 (so the caller can record sparsity), else 0.
__device__ __forceinline__ bool epi_store(const GemmSeg &s, int n, int b, float acc) {
    size_t o = (size_t)b * s.ldo + n;
    switch (s.epi) {
        case EPI_F32: ((float *)s.out)[o] = acc; break;
        case EPI_F16: ((__half *)s.out)[o] = __float2half_rn(acc); break;
        case EPI_F16_TANH: ((__half *)s.out)[o] = __float2half_rn(tanhf(acc)); break;
        case EPI_F16_SIGMOID: ((__half *)s.out)[o] = __float2half_rn(sigm(acc)); break;
        case EPI_DECAY: {
            float t = __half2float(s.bias[n]) + acc;
            ((float *)s.out)[o] = expf(-0.606530659712633f * sigm(t));
            break;
        }
        case EPI_SIGMOID_BIAS: ((float *)s.out)[o] = sigm(__half2float(s.bias[n]) + acc); break;
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

// ---------------------------------------------------------------------------
// Work partition: units (tile, k-block) numbered tile-major; CTA c owns
// [start(c), start(c+1)).
// ---------------------------------------------------------------------------
__device__ __forceinline__ int unit_start(int c, int G, int U) { return (int)(((long long)c * U) / G); }
__device__ __forceinline__ int cta_of_unit(int u, int G, int U) {
    return (int)((((long long)(u + 1)) * G + U - 1) / U) - 1;
}

struct Loc {
    int s, tin, kblk, tile;  // segment, tile within segment, k-block, global tile
};
__device__ __forceinline__ Loc locate(const GemmParams &p, int u) {
    int s = 0;
    while (s + 1 < p.nseg && u >= p.seg[s + 1].unit0) ++s;
    int r = u - p.seg[s].unit0;
    int kb = p.seg[s].kb;
    Loc l;
    l.s = s;
    l.tin = r / kb;
    l.kblk = r - l.tin * kb;
    l.tile = p.seg[s].tile0 + l.tin;
    return l;
}
__device__ __forceinline__ bool unit_skipped(const GemmParams &p, int kblk) {
    return p.nz_skip != nullptr && p.nz_skip[kblk] == 0u;
}

constexpr uint32_t W_TILE_BYTES = GEMM_TILE_M * GEMM_TILE_K * 2;  // 16 KB

__global__ void __launch_bounds__(192, 1) gemm_tc_kernel(const __grid_constant__ GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int S = p.stages;
    const uint32_t XB = (uint32_t)p.npad * 128u;
    uint8_t *sW = base;
    uint8_t *sX = base + (size_t)S * W_TILE_BYTES;
    uint64_t *full = (uint64_t *)(sX + (size_t)S * XB);
    uint64_t *empty = full + S;
    uint64_t *acc_full = empty + S;
    uint64_t *acc_empty = acc_full + 1;
    uint32_t *tmem_slot = (uint32_t *)(acc_empty + 1);
    volatile uint32_t *abort_flag = tmem_slot + 1;
    volatile uint32_t *ticket_s = tmem_slot + 2;
    volatile uint32_t *nzq = tmem_slot + 3;  // [4]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, c = blockIdx.x, U = p.nunits;
    const int u_begin = unit_start(c, G, U), u_end = unit_start(c + 1, G, U);
    uint32_t ncols = 32;
    while ((int)ncols < p.npad) ncols <<= 1;

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 128);
        *abort_flag = 0u;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        for (int i = 0; i < p.nmaps; ++i) prefetch_tmap(&p.maps[i]);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, ncols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t polW = policy_evict_first(), polX = policy_evict_last();
            int npre = 0;
            if (p.prefetch) {
                for (int u = u_begin; u < u_end && npre < S; ++u, ++npre) {
                    Loc l = locate(p, u);
                    const GemmSeg &sg = p.seg[l.s];
                    mbar_expect_tx(&full[npre], W_TILE_BYTES + XB);
                    tma_load_3d(sW + (size_t)npre * W_TILE_BYTES, &p.maps[sg.wmap], &full[npre],
                                l.kblk * GEMM_TILE_K, l.tin * GEMM_TILE_M, sg.layer, polW);
                }
            }
            pdl_wait();
            pdl_launch();
            for (int j = 0; j < npre; ++j) {
                Loc l = locate(p, u_begin + j);
                const GemmSeg &sg = p.seg[l.s];
                for (int r = 0; r < p.npad; r += 16)
                    tma_load_2d(sX + (size_t)j * XB + (size_t)r * 128, &p.maps[sg.xmap], &full[j],
                                l.kblk * GEMM_TILE_K, r, polX);
            }
            int i = npre;
            for (int u = u_begin + npre; u < u_end; ++u) {
                Loc l = locate(p, u);
                if (unit_skipped(p, l.kblk)) continue;
                const GemmSeg &sg = p.seg[l.s];
                const int st = i % S;
                if (i >= S && !mbar_wait(&empty[st], (uint32_t)((i / S) - 1) & 1u, abort_flag)) {
                    *abort_flag = 1u;
                    atomicOr(p.err, ERR_TIMEOUT);
                    break;
                }
                mbar_expect_tx(&full[st], W_TILE_BYTES + XB);
                tma_load_3d(sW + (size_t)st * W_TILE_BYTES, &p.maps[sg.wmap], &full[st], l.kblk * GEMM_TILE_K,
                            l.tin * GEMM_TILE_M, sg.layer, polW);
                for (int r = 0; r < p.npad; r += 16)
                    tma_load_2d(sX + (size_t)st * XB + (size_t)r * 128, &p.maps[sg.xmap], &full[st],
                                l.kblk * GEMM_TILE_K, r, polX);
                ++i;
            }
            // Before leaving, make sure no copy issued by this CTA is still in flight
            // (bounded: the last S stages).
            for (int j = (i > S ? i - S : 0); j < i; ++j) {
                if (!mbar_wait(&full[j % S], (uint32_t)(j / S) & 1u, abort_flag)) break;
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            pdl_wait();
            const uint32_t idesc = idesc_f16(GEMM_TILE_M, p.npad);
            int i = 0, range = 0;
            int u = u_begin;
            bool ok = true;
            while (u < u_end && ok) {
                Loc l = locate(p, u);
                const GemmSeg &sg = p.seg[l.s];
                int r_end = sg.unit0 + (l.tin + 1) * sg.kb;
                if (r_end > u_end) r_end = u_end;
                if (range > 0 && !mbar_wait(acc_empty, (uint32_t)(range - 1) & 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t issued = 0;
                for (; u < r_end; ++u) {
                    int kblk = locate(p, u).kblk;
                    if (unit_skipped(p, kblk)) continue;
                    const int st = i % S;
                    if (!mbar_wait(&full[st], (uint32_t)(i / S) & 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(sW + (size_t)st * W_TILE_BYTES);
                    const uint32_t b0 = smem_u32(sX + (size_t)st * XB);
#pragma unroll
                    for (int kk = 0; kk < GEMM_TILE_K / 16; ++kk)
                        mma_f16(tmem, sdesc_k128(a0 + kk * 32), sdesc_k128(b0 + kk * 32), idesc,
                                (issued | (uint32_t)kk) ? 1u : 0u);
                    issued = 1;
                    mma_commit(&empty[st]);
                    ++i;
                }
                if (!ok) break;
                if (issued)
                    mma_commit(acc_full);
                else
                    mbar_arrive(acc_full);
                ++range;
            }
            if (!ok) {
                *abort_flag = 1u;
                atomicOr(p.err, ERR_TIMEOUT);
            }
        }
    } else {
        // ------------------------------------------------ epilogue (warps 2..5)
        pdl_wait();
        const int q = warp & 3;               // TMEM lane quarter of this warp
        const int row = q * 32 + lane;        // accumulator row = weight row within the tile
        const int et = threadIdx.x - 64;      // 0..127
        const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16);
        int range = 0;
        int u = u_begin;
        while (u < u_end) {
            Loc l = locate(p, u);
            const GemmSeg &sg = p.seg[l.s];
            const int tile_u0 = sg.unit0 + l.tin * sg.kb;
            int r_end = tile_u0 + sg.kb;
            const bool complete = (u == tile_u0) && (r_end <= u_end);
            if (r_end > u_end) r_end = u_end;
            bool valid = false;
            for (int uu = u; uu < r_end; ++uu)
                if (!unit_skipped(p, uu - tile_u0)) valid = true;
            if (!mbar_wait(acc_full, (uint32_t)range & 1u, abort_flag)) {
                *abort_flag = 1u;
                atomicOr(p.err, ERR_TIMEOUT);
                break;
            }
            tc_fence_after();
            const int n = l.tin * GEMM_TILE_M + row;
            bool nzany = false;
            if (complete) {
                for (int cb = 0; cb < p.npad; cb += 16) {
                    float v[16];
                    if (valid) {
                        tmem_ld16(taddr + (uint32_t)cb, v);
                    } else {
#pragma unroll
                        for (int j = 0; j < 16; ++j) v[j] = 0.0f;
                    }
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int b = cb + j;
                        if (b < p.B && n < sg.rows) nzany |= epi_store(sg, n, b, v[j]);
                    }
                }
                tc_fence_before();
                mbar_arrive(acc_empty);
            } else {
                const int first_tile = locate(p, u_begin).tile;
                const int myslot = (l.tile == first_tile) ? 0 : 1;
                float *wsp = p.ws + ((size_t)(c * 2 + myslot) * p.npad) * GEMM_TILE_M;
                for (int cb = 0; cb < p.npad; cb += 16) {
                    float v[16];
                    if (valid) {
                        tmem_ld16(taddr + (uint32_t)cb, v);
                    } else {
#pragma unroll
                        for (int j = 0; j < 16; ++j) v[j] = 0.0f;
                    }
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int b = cb + j;
                        if (b < p.B) __stcg(&wsp[(size_t)b * GEMM_TILE_M + row], v[j]);
                    }
                }
                tc_fence_before();
                mbar_arrive(acc_empty);
                __threadfence();
                named_bar(1, 128);
                if (et == 0) *ticket_s = atomicAdd(&p.counters[l.tile], 1u);
                named_bar(1, 128);
                const int c_first = cta_of_unit(tile_u0, G, U);
                const int c_last = cta_of_unit(tile_u0 + sg.kb - 1, G, U);
                const uint32_t ncontrib = (uint32_t)(c_last - c_first + 1);
                if (*ticket_s == ncontrib - 1u) {
                    __threadfence();
                    for (int b = 0; b < p.B; ++b) {
                        float acc = 0.0f;
                        for (int cc = c_first; cc <= c_last; ++cc) {
                            const int ft = locate(p, unit_start(cc, G, U)).tile;
                            const int sl = (ft == l.tile) ? 0 : 1;
                            acc += __ldcg(&p.ws[((size_t)(cc * 2 + sl) * p.npad + b) * GEMM_TILE_M + row]);
                        }
                        if (n < sg.rows) nzany |= epi_store(sg, n, b, acc);
                    }
                    if (et == 0) p.counters[l.tile] = 0u;
                } else {
                    ++range;
                    u = r_end;
                    continue;  // another CTA finalises this tile
                }
            }
            if (sg.epi == EPI_RELU2 && p.nz_out != nullptr) {
                const unsigned bal = __ballot_sync(0xffffffffu, nzany);
                if (lane == 0) nzq[q] = bal ? 1u : 0u;
                named_bar(2, 128);
                if (et == 0) {
                    const int blk0 = l.tin * 2;
                    const int nblk = (sg.rows + 63) / 64;
                    if (blk0 < nblk) p.nz_out[blk0] = nzq[0] | nzq[1];
                    if (blk0 + 1 < nblk) p.nz_out[blk0 + 1] = nzq[2] | nzq[3];
                }
                named_bar(2, 128);
            }
            ++range;
            u = r_end;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, ncols);
    }
}

size_t gemm_tc_smem_bytes(int npad, int stages) {
    return 1024 + (size_t)stages * (W_TILE_BYTES + (size_t)npad * 128) + (size_t)(2 * stages + 2) * 8 + 64;
}

int gemm_tc_max_smem() { return 227 * 1024; }

void launch_gemm_tc(const GemmParams &p, int grid, size_t smem, const LaunchCfg &lc, cudaError_t *e) {
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t r = cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             gemm_tc_max_smem());
        if (r != cudaSuccess) {
            *e = r;
            return;
        }
        attr_set = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(192);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = lc.stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = lc.pdl ? 1 : 0;
    cudaError_t r = cudaLaunchKernelEx(&cfg, gemm_tc_kernel, p);
    if (r != cudaSuccess) *e = r;
}

// ---------------------------------------------------------------------------
// SIMT cross-check kernel: CTA = 64 output rows of one segment, warp = 8 rows.
// seg.tile0 holds the segment's first 64-row block.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) gemm_simt_kernel(const __grid_constant__ GemmParams p) {
    __shared__ uint32_t nzw[8];
    int s = 0;
    while (s + 1 < p.nseg && (int)blockIdx.x >= p.seg[s + 1].tile0) ++s;
    const GemmSeg &sg = p.seg[s];
    const int blk = blockIdx.x - sg.tile0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_wait();
    pdl_launch();
    bool nzany = false;
    for (int rr = 0; rr < 8; ++rr) {
        const int n = blk * 64 + warp * 8 + rr;
        if (n >= sg.rows) break;
        const __half *wrow = sg.w + (size_t)n * sg.K;
        for (int b0 = 0; b0 < p.B; b0 += 8) {
            float acc[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
            for (int k = lane * 8; k < sg.K; k += 256) {
                if (unit_skipped(p, k / GEMM_TILE_K)) continue;
                const uint4 wv = *(const uint4 *)(wrow + k);
                const __half2 *w2 = (const __half2 *)&wv;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (b0 + j < p.B) {
                        const uint4 xv = *(const uint4 *)(sg.x + (size_t)(b0 + j) * sg.ldx + k);
                        const __half2 *x2 = (const __half2 *)&xv;
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            float2 wf = __half22float2(w2[t]), xf = __half22float2(x2[t]);
                            acc[j] = fmaf(wf.x, xf.x, acc[j]);
                            acc[j] = fmaf(wf.y, xf.y, acc[j]);
                        }
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] = warp_sum(acc[j]);
            if (lane < 8 && b0 + lane < p.B) {
                float v = acc[0];
#pragma unroll
                for (int j = 1; j < 8; ++j)
                    if (lane == j) v = acc[j];
                nzany |= epi_store(sg, n, b0 + lane, v);
            }
        }
    }
    if (sg.epi == EPI_RELU2 && p.nz_out != nullptr) {
        const unsigned bal = __ballot_sync(0xffffffffu, nzany);
        if (lane == 0) nzw[warp] = bal ? 1u : 0u;
        __syncthreads();
        if (threadIdx.x == 0) {
            uint32_t f = 0;
            for (int w = 0; w < 8; ++w) f |= nzw[w];
            p.nz_out[blk] = f;
        }
    }
}

void launch_gemm_simt(const GemmParams &p, const LaunchCfg &lc, cudaError_t *e) {
    int nblk = 0;
    for (int s = 0; s < p.nseg; ++s) nblk += (p.seg[s].rows + 63) / 64;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(nblk);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = lc.stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = lc.pdl ? 1 : 0;
    cudaError_t r = cudaLaunchKernelEx(&cfg, gemm_simt_kernel, p);
    if (r != cudaSuccess) *e = r;
}

}  // namespace rk
