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
//    loads of 16 KB weight tiles (stored contiguously, so each load is one
//    sequential 16 KB read) and Bx64 activation tiles into a ring of
//    shared-memory stages, warp 1 issues tcgen05.mma into a TMEM accumulator
//    (two buffers when they fit, so the next item's MMAs overlap the previous
//    epilogue), warps 2-5 drain TMEM and apply the epilogue.  Work items are
//    (row tile, k-range) pairs split evenly over the grid; a split k-range
//    stores fp32 partial sums that the consuming kernel adds in a fixed order,
//    so no CTA waits for another and results do not depend on timing.
//  * SIMT kernel: a plain warp-per-row dot product with the same epilogues and
//    partial layout, kept as an independent cross-check of the tensor-core kernel.
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
                                        int B, int c0) {
    const bool live = n < sg.rows;
    float bias = 0.0f;
    if ((KIND == EPI_DECAY || KIND == EPI_SIGMOID_BIAS) && live) bias = __half2float(sg.bias[n]);
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

__device__ __forceinline__ bool epi_item(const GemmSeg &sg, uint32_t taddr, bool valid, int n, int split, int npad,
                                         int B, int c0) {
    if (sg.S > 1) return epi_run<-1>(sg, taddr, valid, n, split, npad, B, c0);
    switch (sg.epi) {
        case EPI_F32: return epi_run<EPI_F32>(sg, taddr, valid, n, split, npad, B, c0);
        case EPI_F16: return epi_run<EPI_F16>(sg, taddr, valid, n, split, npad, B, c0);
        case EPI_F16_TANH: return epi_run<EPI_F16_TANH>(sg, taddr, valid, n, split, npad, B, c0);
        case EPI_F16_SIGMOID: return epi_run<EPI_F16_SIGMOID>(sg, taddr, valid, n, split, npad, B, c0);
        case EPI_DECAY: return epi_run<EPI_DECAY>(sg, taddr, valid, n, split, npad, B, c0);
        case EPI_SIGMOID_BIAS: return epi_run<EPI_SIGMOID_BIAS>(sg, taddr, valid, n, split, npad, B, c0);
        case EPI_RESID: return epi_run<EPI_RESID>(sg, taddr, valid, n, split, npad, B, c0);
        case EPI_RELU2: return epi_run<EPI_RELU2>(sg, taddr, valid, n, split, npad, B, c0);
        default: return false;
    }
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


__global__ void __launch_bounds__(GEMM_TC_THREADS, 1) gemm_tc_kernel(const __grid_constant__ GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    // Segment descriptors and sparsity flags are staged in shared memory and the
    // scalars in registers: the parameter block is only addressed for the tensor
    // maps, so nothing in the loops re-reads it.
    __shared__ GemmSeg sseg[GEMM_MAX_SEG];
    __shared__ uint32_t snz[MAX_NZ_BLOCKS];
    __shared__ uint64_t flags_ready;
    __shared__ uint32_t s_ok;
    uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int S = p.stages, B = p.B, npad = p.npad, NB = p.accbufs, nseg = p.nseg, nitems = p.nitems;
    const bool has_skip = p.nz_skip != nullptr;
    const uint32_t *skip = has_skip ? snz : nullptr;
    const uint32_t XKB = (uint32_t)npad * 128u;  // one activation k-block
    const uint32_t XB = KB_STAGE * XKB;            // per stage
    uint8_t *sW = base;
    uint8_t *sX = base + (size_t)S * W_STAGE_BYTES;
    uint64_t *full = (uint64_t *)(sX + (size_t)S * XB);
    uint64_t *empty = full + S;
    uint64_t *acc_full = empty + S;      // [2]
    uint64_t *acc_empty = acc_full + 2;  // [2]
    uint32_t *tmem_slot = (uint32_t *)(acc_empty + 2);
    volatile uint32_t *abort_flag = tmem_slot + 1;
    uint32_t *nzf = tmem_slot + 2;  // [2]: some output of tile rows 0-63 / 64-127 was nonzero

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, c = blockIdx.x;
    const int i_begin = item_first(c, G, nitems), i_end = item_first(c + 1, G, nitems);
    uint32_t ncols = 32;
    while ((int)ncols < NB * npad) ncols <<= 1;

    if (threadIdx.x < nseg) sseg[threadIdx.x] = p.seg[threadIdx.x];
    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], EPI_THREADS);
        }
        mbar_init(&flags_ready, 1);
        *abort_flag = 0u;
        nzf[0] = nzf[1] = 0u;
        fence_barrier_init();
    }
    __syncthreads();

    // Weight prefetch before the dependency wait (weights are constant), issued
    // before the TMEM allocation so it proceeds even while a predecessor's CTA
    // still holds tensor memory on this SM.
    int npre = 0;
    if (warp == 0 && lane == 0) {
        for (int i = 0; i < p.nmaps; ++i) prefetch_tmap(&p.maps[i]);
        if (p.prefetch) {
            const uint64_t polW = policy_evict_first();
            for (int i = i_begin; i < i_end && npre < S; ++i) {
                const Item it = locate_item(sseg, nseg, i);
                const int tb = sseg[it.s].tile_base + it.tile * sseg[it.s].kb;
                const CUtensorMap *wm = &p.maps[sseg[it.s].wmap];
                for (int kb = it.kb0; kb < it.kb1 && npre < S; kb += KB_STAGE, ++npre) {
                    mbar_expect_tx(&full[npre], W_STAGE_BYTES + XB);
                    tma_load_3d(sW + (size_t)npre * W_STAGE_BYTES, wm, &full[npre], 0, 0, tb + kb, polW);
                }
            }
        }
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
            pdl_wait();
            pdl_launch();
            bool ok = true;
            if (has_skip && !mbar_wait(&flags_ready, 0u, abort_flag)) ok = false;
            int q = 0;  // stage sequence number
            for (int i = i_begin; i < i_end && ok; ++i) {
                const Item it = locate_item(sseg, nseg, i);
                const int tb = sseg[it.s].tile_base + it.tile * sseg[it.s].kb;
                const CUtensorMap *wm = &p.maps[sseg[it.s].wmap];
                const CUtensorMap *xm = &p.maps[sseg[it.s].xmap];
                for (int kb = it.kb0; kb < it.kb1; kb += KB_STAGE) {
                    if (stage_skipped(skip, kb)) continue;
                    const int st = q % S;
                    if (q >= npre) {
                        if (q >= S && !mbar_wait(&empty[st], (uint32_t)((q / S) - 1) & 1u, abort_flag)) {
                            ok = false;
                            break;
                        }
                        mbar_expect_tx(&full[st], W_STAGE_BYTES + XB);
                        tma_load_3d(sW + (size_t)st * W_STAGE_BYTES, wm, &full[st], 0, 0, tb + kb, polW);
                    }  // else: the weights were requested before the dependency wait
                    if (sseg[it.s].x3) {
                        tma_load_3d(sX + (size_t)st * XB, xm, &full[st], 0, 0, kb, polX);
                    } else {
#pragma unroll
                        for (int h = 0; h < KB_STAGE; ++h)
                            tma_load_2d(sX + (size_t)st * XB + (size_t)h * XKB, xm, &full[st], (kb + h) * GEMM_TILE_K,
                                        0, polX);
                    }
                    ++q;
                }
            }
            if (!ok) {
                *abort_flag = 1u;
                atomicOr(p.err, ERR_TIMEOUT);
            }
            // Before leaving, wait (bounded) until no copy issued here is in flight.
            for (int j = (q > S ? q - S : 0); j < q; ++j)
                if (!mbar_wait(&full[j % S], (uint32_t)(j / S) & 1u, abort_flag)) break;
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_f16(GEMM_TILE_M, npad);
            bool ok = true;
            if (has_skip && !mbar_wait(&flags_ready, 0u, abort_flag)) ok = false;
            int q = 0, n = 0;
            for (int i = i_begin; i < i_end && ok; ++i, ++n) {
                const Item it = locate_item(sseg, nseg, i);
                const int buf = n % NB;
                if (n >= NB && !mbar_wait(&acc_empty[buf], (uint32_t)((n / NB) - 1) & 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem + (uint32_t)(buf * npad);
                uint32_t issued = 0;
                for (int kb = it.kb0; kb < it.kb1; kb += KB_STAGE) {
                    if (stage_skipped(skip, kb)) continue;
                    const int st = q % S;
                    if (!mbar_wait(&full[st], (uint32_t)(q / S) & 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(sW + (size_t)st * W_STAGE_BYTES);
                    const uint32_t b0 = smem_u32(sX + (size_t)st * XB);
#pragma unroll
                    for (int kk = 0; kk < KB_STAGE * GEMM_TILE_K / 16; ++kk)
                        mma_f16(d_tmem, sdesc_k128(a0 + (kk >> 2) * W_TILE_BYTES + (kk & 3) * 32),
                                sdesc_k128(b0 + (kk >> 2) * XKB + (kk & 3) * 32), idesc, (issued | (uint32_t)kk) ? 1u : 0u);
                    issued = 1;
                    mma_commit(&empty[st]);
                    ++q;
                }
                if (!ok) break;
                if (issued)
                    mma_commit(&acc_full[buf]);
                else
                    mbar_arrive(&acc_full[buf]);
            }
            if (!ok) {
                *abort_flag = 1u;
                atomicOr(p.err, ERR_TIMEOUT);
            }
        }
    } else {
        // ------------------------------------------------ epilogue (warps 2..5)
        pdl_wait();
        const int qd = warp & 3;              // TMEM lane quarter of this warp
        const int row = qd * 32 + lane;       // accumulator row = weight row within the tile
        const int et = threadIdx.x - 64;      // 0..EPI_THREADS-1
        const int grp = et >> 7;              // column-chunk group within the lane quarter
        uint32_t *nz_out = p.nz_out;
        if (has_skip) {  // stage the k-block flags written by the preceding kernel
            const int nkb = sseg[0].kb < MAX_NZ_BLOCKS ? sseg[0].kb : MAX_NZ_BLOCKS;  // padded count
            const int nreal = (sseg[0].K + GEMM_TILE_K - 1) / GEMM_TILE_K;             // flags written
            for (int j = et; j < nkb; j += EPI_THREADS) snz[j] = j < nreal ? p.nz_skip[j] : 0u;
            named_bar(1, EPI_THREADS);
            if (et == 0) mbar_arrive(&flags_ready);
        }
        int n = 0;
        for (int i = i_begin; i < i_end; ++i, ++n) {
            const Item it = locate_item(sseg, nseg, i);
            const GemmSeg sg = sseg[it.s];  // register copy
            const int buf = n % NB;
            bool valid = false;
            for (int kb = it.kb0; kb < it.kb1; kb += KB_STAGE)
                if (!stage_skipped(skip, kb)) valid = true;
            // thread 0 waits and tells the others, so that all 128 threads take
            // the same path through the named barriers below
            if (et == 0) s_ok = mbar_wait(&acc_full[buf], (uint32_t)(n / NB) & 1u, abort_flag) ? 1u : 0u;
            named_bar(3, EPI_THREADS);
            const bool ok_wait = s_ok != 0u;
            named_bar(3, EPI_THREADS);
            if (!ok_wait) {
                if (et == 0) {
                    *abort_flag = 1u;
                    atomicOr(p.err, ERR_TIMEOUT);
                }
                break;
            }
            (void)mbar_try_wait(&acc_full[buf], (uint32_t)(n / NB) & 1u);
            tc_fence_after();
            const uint32_t taddr = tmem + ((uint32_t)(qd * 32) << 16) + (uint32_t)(buf * npad);
            const int nrow = it.tile * GEMM_TILE_M + row;
            const bool nzany = epi_item(sg, taddr, valid, nrow, it.split, npad, B, grp * EPI_CW);
            tc_fence_before();
            mbar_arrive(&acc_empty[buf]);
            if (sg.epi == EPI_RELU2 && sg.S == 1 && nz_out != nullptr) {
                const unsigned bal = __ballot_sync(0xffffffffu, nzany);
                if (lane == 0 && bal) atomicOr(&nzf[qd >> 1], 1u);
                named_bar(2, EPI_THREADS);
                if (et == 0) {
                    const int blk0 = it.tile * 2;
                    const int nblk = (sg.rows + 63) / 64;
                    const uint32_t f0 = ((volatile uint32_t *)nzf)[0], f1 = ((volatile uint32_t *)nzf)[1];
                    nzf[0] = nzf[1] = 0u;  // for the next item, after the barrier below
                    if (blk0 < nblk) nz_out[blk0] = f0;
                    if (blk0 + 1 < nblk) nz_out[blk0 + 1] = f1;
                    const unsigned long long nnz = (blk0 < nblk ? f0 : 0u) + (blk0 + 1 < nblk ? f1 : 0u);
                    if (p.nz_count && nnz) atomicAdd(p.nz_count, nnz);
                }
                named_bar(2, EPI_THREADS);
            }
        }
    }

    __syncwarp();  // warps 0 and 1 reconverge (lane 0 ran the producer / MMA loop)
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, ncols);
    }
}

// ---------------------------------------------------------------------------
// int8-weight variant.  A weight tile arrives as 128 rows x 64 int8 (8 KB; the
// int8 tiles keep the fp16 tile order), is widened to fp16 in registers and
// stored into tensor memory, from where tcgen05.mma kind::f16 reads it as the
// A operand; the row scale multiplies the finished sum in the epilogue (W = q *
// scale per row, so W x = scale * (q x)).
// Shared memory: ring W (SA stages of the int8 tiles of kbs k-blocks, TMA with
// the 64-byte swizzle: 16-byte chunk c of row r at c ^ ((r >> 1) & 3), so that
// a warp reading one chunk of 32 rows hits every bank once) and ring X (SX
// stages of activation boxes).  Tensor memory: the accumulators and SB = 4
// stages of widened weights (kbs x 32 columns each).
// Roles: warp 0 lane 0 streams ring W from the first instant (weights are
// constant: no dependency wait); warp 18 lane 0 loads ring X after the
// dependency wait; warp 1 lane 0 issues the MMAs; the 16 epilogue warps form
// four groups of four (one warp per TMEM lane quarter = 32 weight rows, one
// row per lane) that widen stages q with q % 4 == group -- four stages in
// flight -- and run the epilogue after each item.  A ring W slot is released
// as soon as its group has widened it, so the int8 stream runs up to SA stages
// ahead of the tensor cores.  SB = 4 and SA a multiple of 4 (chosen by the
// host): a slot's previous stage then belongs to the same group, which has
// already waited on it, so no barrier is ever waited on two phases ahead.
// Barriers: full_w / empty_w (int8 bytes landed / the group's 4 warps),
// full_x / empty_x (activation bytes landed / the MMA commit), full_b (the
// group's 4 warps) / empty_b (the MMA commit).
// ---------------------------------------------------------------------------
constexpr uint32_t W8_TILE_BYTES = GEMM_TILE_M * GEMM_TILE_K;  // 8 KB
constexpr int CONV_GROUPS = EPI_WARPS / 4;
constexpr int GEMM_TC8_THREADS = GEMM_TC_THREADS + 32;          // + the activation producer warp
constexpr int XPROD_WARP = GEMM_TC_THREADS / 32;

// 16 int8 -> 8 words of two fp16 each (element 2j in the low half of word j).
// Exact: the byte x ^ 0x80 = x + 128 is placed in the low mantissa byte of the
// fp16 1024.0 (0x6400), giving 1024 + 128 + x, and 1152 is subtracted.
__device__ __forceinline__ void widen16(const uint4 in, uint32_t *o) {
    const uint32_t w[4] = {in.x, in.y, in.z, in.w};
    const __half2 off = __halves2half2(__ushort_as_half((unsigned short)0x6480u),
                                       __ushort_as_half((unsigned short)0x6480u));  // 1152
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t u = w[k] ^ 0x80808080u;
        const uint32_t lo = __byte_perm(u, 0x64646464u, 0x5140u);
        const uint32_t hi = __byte_perm(u, 0x64646464u, 0x5342u);
        __half2 hl = __hsub2(*reinterpret_cast<const __half2 *>(&lo), off);
        __half2 hh = __hsub2(*reinterpret_cast<const __half2 *>(&hi), off);
        o[2 * k] = *reinterpret_cast<uint32_t *>(&hl);
        o[2 * k + 1] = *reinterpret_cast<uint32_t *>(&hh);
    }
}

__device__ __forceinline__ bool stage_skipped_k(const uint32_t *flags, int kb, int kbs) {
    return flags != nullptr && flags[kb] == 0u && (kbs == 1 || flags[kb + 1] == 0u);
}

__global__ void __launch_bounds__(GEMM_TC8_THREADS, 1) gemm_tc8_kernel(const __grid_constant__ GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ GemmSeg sseg[GEMM_MAX_SEG];
    __shared__ uint32_t snz[MAX_NZ_BLOCKS];
    __shared__ uint64_t flags_ready;
    __shared__ uint32_t s_ok;
    uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int SA = p.stages, SB = p.stages_b, SX = p.stages_x, KBS = p.kbs;
    const int B = p.B, npad = p.npad, NB = p.accbufs, nseg = p.nseg, nitems = p.nitems;
    const bool has_skip = p.nz_skip != nullptr;
    const uint32_t *skip = has_skip ? snz : nullptr;
    const uint32_t XKB = (uint32_t)npad * 128u;        // one activation k-block
    const uint32_t W8B = (uint32_t)KBS * W8_TILE_BYTES;  // ring W stage (a multiple of 1024)
    const uint32_t XB = (uint32_t)KBS * XKB;            // ring X stage (a multiple of 1024)
    uint8_t *sW = base;
    uint8_t *sX = base + (size_t)SA * W8B;
    uint64_t *full_w = (uint64_t *)(sX + (size_t)SX * XB);
    uint64_t *empty_w = full_w + SA;
    uint64_t *full_x = empty_w + SA;
    uint64_t *empty_x = full_x + SX;
    uint64_t *full_b = empty_x + SX;
    uint64_t *empty_b = full_b + SB;
    uint64_t *acc_full = empty_b + SB;   // [2]
    uint64_t *acc_empty = acc_full + 2;  // [2]
    uint32_t *tmem_slot = (uint32_t *)(acc_empty + 2);
    volatile uint32_t *abort_flag = tmem_slot + 1;
    uint32_t *nzf = tmem_slot + 2;  // [2]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, c = blockIdx.x;
    const int i_begin = item_first(c, G, nitems), i_end = item_first(c + 1, G, nitems);
    const uint32_t ncols = 512;                        // accumulators + widened weight stages
    const uint32_t acol0 = (uint32_t)(NB * npad);      // first column of the weight stages

    if (threadIdx.x < nseg) sseg[threadIdx.x] = p.seg[threadIdx.x];
    if (threadIdx.x == 0) {
        for (int i = 0; i < SA; ++i) {
            mbar_init(&full_w[i], 1);
            mbar_init(&empty_w[i], 4);
        }
        for (int i = 0; i < SX; ++i) {
            mbar_init(&full_x[i], 1);
            mbar_init(&empty_x[i], 1);
        }
        for (int i = 0; i < SB; ++i) {
            mbar_init(&full_b[i], 4);
            mbar_init(&empty_b[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], EPI_THREADS);
        }
        mbar_init(&flags_ready, 1);
        *abort_flag = 0u;
        nzf[0] = nzf[1] = 0u;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0)
        for (int i = 0; i < p.nmaps; ++i) prefetch_tmap(&p.maps[i]);
    if (warp == 1) {
        tmem_alloc(tmem_slot, ncols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------ int8 weight producer (ring W)
        if (lane == 0) {
            const uint64_t polW = policy_evict_first();
            bool ok = true;
            // the skipped stages depend on flags the preceding kernel writes
            if (has_skip && !mbar_wait(&flags_ready, 0u, abort_flag)) ok = false;
            int q = 0;
            for (int i = i_begin; i < i_end && ok; ++i) {
                const Item it = locate_item(sseg, nseg, i);
                const int tb = sseg[it.s].tile_base + it.tile * sseg[it.s].kb;
                const CUtensorMap *wm = &p.maps[sseg[it.s].wmap];
                for (int kb = it.kb0; kb < it.kb1; kb += KBS) {
                    if (stage_skipped_k(skip, kb, KBS)) continue;
                    const int st = q % SA;
                    if (q >= SA && !mbar_wait(&empty_w[st], (uint32_t)((q / SA) - 1) & 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(&full_w[st], W8B);
                    tma_load_3d(sW + (size_t)st * W8B, wm, &full_w[st], 0, 0, tb + kb, polW);
                    ++q;
                }
            }
            if (!ok) {
                *abort_flag = 1u;
                atomicOr(p.err, ERR_TIMEOUT);
            }
            // before leaving, wait (bounded) until no copy issued here is in flight
            for (int j = (q > SA ? q - SA : 0); j < q; ++j)
                if (!mbar_wait_any(&full_w[j % SA], (uint32_t)(j / SA) & 1u)) break;
        }
    } else if (warp == XPROD_WARP) {
        // ------------------------------------------------ activation producer (ring X)
        if (lane == 0) {
            const uint64_t polX = policy_evict_last();
            pdl_wait();
            pdl_launch();
            bool ok = true;
            if (has_skip && !mbar_wait(&flags_ready, 0u, abort_flag)) ok = false;
            int q = 0;
            for (int i = i_begin; i < i_end && ok; ++i) {
                const Item it = locate_item(sseg, nseg, i);
                const CUtensorMap *xm = &p.maps[sseg[it.s].xmap];
                for (int kb = it.kb0; kb < it.kb1; kb += KBS) {
                    if (stage_skipped_k(skip, kb, KBS)) continue;
                    const int st = q % SX;
                    if (q >= SX && !mbar_wait(&empty_x[st], (uint32_t)((q / SX) - 1) & 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    uint8_t *sx = sX + (size_t)st * XB;
                    mbar_expect_tx(&full_x[st], XB);
                    if (sseg[it.s].x3) {
                        tma_load_3d(sx, xm, &full_x[st], 0, 0, kb, polX);
                    } else {
                        for (int h = 0; h < KBS; ++h)
                            tma_load_2d(sx + (size_t)h * XKB, xm, &full_x[st], (kb + h) * GEMM_TILE_K, 0, polX);
                    }
                    ++q;
                }
            }
            if (!ok) {
                *abort_flag = 1u;
                atomicOr(p.err, ERR_TIMEOUT);
            }
            for (int j = (q > SX ? q - SX : 0); j < q; ++j)
                if (!mbar_wait_any(&full_x[j % SX], (uint32_t)(j / SX) & 1u)) break;
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_f16(GEMM_TILE_M, npad);
            bool ok = true;
            if (has_skip && !mbar_wait(&flags_ready, 0u, abort_flag)) ok = false;
            int q = 0, n = 0;
            for (int i = i_begin; i < i_end && ok; ++i, ++n) {
                const Item it = locate_item(sseg, nseg, i);
                const int buf = n % NB;
                if (n >= NB && !mbar_wait(&acc_empty[buf], (uint32_t)((n / NB) - 1) & 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem + (uint32_t)(buf * npad);
                uint32_t issued = 0;
                for (int kb = it.kb0; kb < it.kb1; kb += KBS) {
                    if (stage_skipped_k(skip, kb, KBS)) continue;
                    const int sx = q % SX, sb = q % SB;
                    if (!mbar_wait(&full_x[sx], (uint32_t)(q / SX) & 1u, abort_flag) ||
                        !mbar_wait(&full_b[sb], (uint32_t)(q / SB) & 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = tmem + acol0 + (uint32_t)(sb * KBS * 32);
                    const uint32_t b0 = smem_u32(sX + (size_t)sx * XB);
                    for (int h = 0; h < KBS; ++h) {
#pragma unroll
                        for (int kk = 0; kk < GEMM_TILE_K / 16; ++kk)
                            mma_f16_ts(d_tmem, a0 + (uint32_t)(h * 32 + kk * 8), sdesc_k128(b0 + h * XKB + kk * 32),
                                       idesc, (issued | (uint32_t)h | (uint32_t)kk) ? 1u : 0u);
                    }
                    issued = 1;
                    mma_commit(&empty_x[sx]);
                    mma_commit(&empty_b[sb]);
                    ++q;
                }
                if (!ok) break;
                if (issued)
                    mma_commit(&acc_full[buf]);
                else
                    mbar_arrive(&acc_full[buf]);
            }
            if (!ok) {
                *abort_flag = 1u;
                atomicOr(p.err, ERR_TIMEOUT);
            }
        }
    } else {
        // ------------------------------------------------ converters + epilogue
        const int qd = warp & 3;              // TMEM lane quarter = weight rows qd*32 .. +31
        const int row = qd * 32 + lane;
        const int et = threadIdx.x - 64;
        const int grp = et >> 7;              // converter group: stages q with q % 4 == grp
        const uint32_t tlane = (uint32_t)(qd * 32) << 16;
        uint32_t *nz_out = p.nz_out;
        bool waited = false;
        if (has_skip) {
            pdl_wait();
            waited = true;
            const int nkb = sseg[0].kb < MAX_NZ_BLOCKS ? sseg[0].kb : MAX_NZ_BLOCKS;
            const int nreal = (sseg[0].K + GEMM_TILE_K - 1) / GEMM_TILE_K;
            for (int j = et; j < nkb; j += EPI_THREADS) snz[j] = j < nreal ? p.nz_skip[j] : 0u;
            named_bar(1, EPI_THREADS);
            if (et == 0) mbar_arrive(&flags_ready);
        }
        int q = 0, n = 0;
        bool ok = true, dead = false;
        for (int i = i_begin; i < i_end && ok; ++i, ++n) {
            const Item it = locate_item(sseg, nseg, i);
            const GemmSeg sg = sseg[it.s];
            const int buf = n % NB;
            bool valid = false;
            for (int kb = it.kb0; kb < it.kb1; kb += KBS) {
                if (stage_skipped_k(skip, kb, KBS)) continue;
                valid = true;
                const int qq = q++;
                if (qq % CONV_GROUPS != grp || dead) continue;  // another group's stage
                const int sa = qq % SA, sb = qq % SB;
                uint32_t w_ok = 0u;
                if (lane == 0) {
                    bool okw = mbar_wait(&full_w[sa], (uint32_t)(qq / SA) & 1u, abort_flag);
                    if (okw && qq >= SB) okw = mbar_wait(&empty_b[sb], (uint32_t)((qq / SB) - 1) & 1u, abort_flag);
                    if (!okw) {
                        *abort_flag = 1u;
                        atomicOr(p.err, ERR_TIMEOUT);
                    }
                    w_ok = okw ? 1u : 0u;
                }
                w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
                if (!w_ok) {
                    dead = true;
                    continue;
                }
                // acquire the landed int8 bytes / the released weight stage in every lane
                (void)mbar_try_wait(&full_w[sa], (uint32_t)(qq / SA) & 1u);
                if (qq >= SB) (void)mbar_try_wait(&empty_b[sb], (uint32_t)((qq / SB) - 1) & 1u);
                tc_fence_after();
                const uint8_t *a8 = sW + (size_t)sa * W8B + row * 64;
                const int sw = (row >> 1) & 3;
                for (int h = 0; h < KBS; ++h) {
                    uint32_t o[32];
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        const uint4 in =
                            *reinterpret_cast<const uint4 *>(a8 + (size_t)h * W8_TILE_BYTES + ((cc ^ sw) << 4));
                        widen16(in, o + 8 * cc);
                    }
                    tmem_st32(tmem + tlane + acol0 + (uint32_t)(sb * KBS * 32 + h * 32), o);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty_w[sa]);  // the int8 bytes are read: the slot may refill
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&full_b[sb]);
            }
            if (!waited) {  // outputs may be read by the preceding kernel until it completes
                pdl_wait();
                waited = true;
            }
            // epilogue of the item (as in gemm_tc_kernel); thread 0 decides for all
            // 512 threads, so that they take the same path through the named barriers
            named_bar(3, EPI_THREADS);
            if (et == 0)
                s_ok = (!*abort_flag && mbar_wait(&acc_full[buf], (uint32_t)(n / NB) & 1u, abort_flag)) ? 1u : 0u;
            named_bar(3, EPI_THREADS);
            const bool ok_wait = s_ok != 0u;
            named_bar(3, EPI_THREADS);
            if (!ok_wait) {
                ok = false;
                break;
            }
            (void)mbar_try_wait(&acc_full[buf], (uint32_t)(n / NB) & 1u);
            tc_fence_after();
            const uint32_t taddr = tmem + tlane + (uint32_t)(buf * npad);
            const int nrow = it.tile * GEMM_TILE_M + row;
            const bool nzany = epi_item(sg, taddr, valid, nrow, it.split, npad, B, grp * EPI_CW);
            tc_fence_before();
            mbar_arrive(&acc_empty[buf]);
            if (sg.epi == EPI_RELU2 && sg.S == 1 && nz_out != nullptr) {
                const unsigned bal = __ballot_sync(0xffffffffu, nzany);
                if (lane == 0 && bal) atomicOr(&nzf[qd >> 1], 1u);
                named_bar(2, EPI_THREADS);
                if (et == 0) {
                    const int blk0 = it.tile * 2;
                    const int nblk = (sg.rows + 63) / 64;
                    const uint32_t f0 = ((volatile uint32_t *)nzf)[0], f1 = ((volatile uint32_t *)nzf)[1];
                    nzf[0] = nzf[1] = 0u;
                    if (blk0 < nblk) nz_out[blk0] = f0;
                    if (blk0 + 1 < nblk) nz_out[blk0 + 1] = f1;
                    const unsigned long long nnz = (blk0 < nblk ? f0 : 0u) + (blk0 + 1 < nblk ? f1 : 0u);
                    if (p.nz_count && nnz) atomicAdd(p.nz_count, nnz);
                }
                named_bar(2, EPI_THREADS);
            }
        }
        if (!ok && et == 0) {
            *abort_flag = 1u;
            atomicOr(p.err, ERR_TIMEOUT);
        }
        if (!waited) pdl_wait();
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, ncols);
    }
}

size_t gemm_tc8_smem_bytes(int npad, int kbs, int stages_w, int stages_x) {
    return 1024 + (size_t)stages_w * kbs * W8_TILE_BYTES + (size_t)stages_x * kbs * npad * 128 +
           (size_t)(2 * stages_w + 2 * stages_x + 2 * 8 + 4) * 8 + 64;
}

void launch_gemm_tc8(const GemmParams &p, int grid, size_t smem, const LaunchCfg &lc, cudaError_t *e) {
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t r = cudaFuncSetAttribute(gemm_tc8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             gemm_tc_max_smem());
        if (r != cudaSuccess) {
            *e = r;
            return;
        }
        attr_set = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(GEMM_TC8_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = lc.stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = lc.pdl ? 1 : 0;
    cudaError_t r = cudaLaunchKernelEx(&cfg, gemm_tc8_kernel, p);  // GEMM_TC8_THREADS threads
    if (r != cudaSuccess) *e = r;
}

size_t gemm_tc_smem_bytes(int npad, int stages) {
    return 1024 + (size_t)stages * (W_STAGE_BYTES + (size_t)KB_STAGE * npad * 128) + (size_t)(2 * stages + 4) * 8 + 64;
}

size_t gemm_tc_stage_bytes(int npad) { return W_STAGE_BYTES + (size_t)KB_STAGE * npad * 128; }

int gemm_tc_max_smem() { return 220 * 1024; }  // dynamic part; static staging takes ~5 KB

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
    cfg.blockDim = dim3(GEMM_TC_THREADS);
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
// SIMT cross-check kernel: CTA = 64 output rows x one split of one segment,
// warp = 8 rows; reads the tiled weight layout directly.  seg.item0 holds the
// segment's first CTA (64-row block x split).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) gemm_simt_kernel(const __grid_constant__ GemmParams p) {
    __shared__ uint32_t nzw[8];
    int s = 0;
    while (s + 1 < p.nseg && (int)blockIdx.x >= p.seg[s + 1].item0) ++s;
    const GemmSeg &sg = p.seg[s];
    const int local = blockIdx.x - sg.item0;
    const int blk = local / sg.S, split = local % sg.S;
    const int kb0 = (int)(((long long)split * sg.kb) / sg.S), kb1 = (int)(((long long)(split + 1) * sg.kb) / sg.S);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_wait();
    pdl_launch();
    bool nzany = false;
    for (int rr = 0; rr < 8; ++rr) {
        const int n = blk * 64 + warp * 8 + rr;
        if (n >= sg.rows) break;
        const int tr = n / GEMM_TILE_M, rin = n % GEMM_TILE_M;
        for (int b0 = 0; b0 < p.B; b0 += 8) {
            float acc[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
            for (int k = kb0 * GEMM_TILE_K + lane * 8; k < kb1 * GEMM_TILE_K && k < sg.K; k += 256) {
                if (kblock_skipped(p.nz_skip, k / GEMM_TILE_K)) continue;
                const __half *wp = sg.w + (((size_t)tr * sg.kb + k / GEMM_TILE_K) * GEMM_TILE_M + rin) * GEMM_TILE_K +
                                   (k % GEMM_TILE_K);
                const uint4 wv = *(const uint4 *)wp;
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
                const int b = b0 + lane;
                if (sg.S > 1) {
                    ((float *)sg.out)[(size_t)split * sg.split_stride + (size_t)b * sg.ldo + n] = v;
                } else if (sg.epi == EPI_RESID) {
                    ((float *)sg.out)[(size_t)b * sg.ldo + n] += v;
                } else {
                    const float bias = (sg.bias != nullptr) ? __half2float(sg.bias[n]) : 0.0f;
                    nzany |= epi_store(sg, n, b, v, bias);
                }
            }
        }
    }
    if (sg.epi == EPI_RELU2 && sg.S == 1 && p.nz_out != nullptr) {
        const unsigned bal = __ballot_sync(0xffffffffu, nzany);
        if (lane == 0) nzw[warp] = bal ? 1u : 0u;
        __syncthreads();
        if (threadIdx.x == 0) {
            uint32_t f = 0;
            for (int w = 0; w < 8; ++w) f |= nzw[w];
            p.nz_out[blk] = f;
            if (p.nz_count && f) atomicAdd(p.nz_count, 1ull);
        }
    }
}

void launch_gemm_simt(const GemmParams &p, const LaunchCfg &lc, cudaError_t *e) {
    int nblk = 0;
    for (int s = 0; s < p.nseg; ++s) nblk += ((p.seg[s].rows + 63) / 64) * p.seg[s].S;
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
