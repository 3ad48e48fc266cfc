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
//    epilogue), 16 epilogue warps drain TMEM and apply the epilogue
//    (gemm_common.cuh).  Work items are
//    (row tile, k-range) pairs split evenly over the grid; a split k-range
//    stores fp32 partial sums that the consuming kernel adds in a fixed order,
//    so results do not depend on timing.  A two-phase launch chains two
//    dependent projections in one grid (every CTA resident): its phase-1
//    activations are read once an in-kernel counter shows the phase-0 items
//    that produce them stored (bounded waits), and a split phase-0 tile may
//    be finished in the launch by its last split (an atomic ticket picks it;
//    it adds the slabs in slab order).
//  * SIMT kernel: a plain warp-per-row dot product with the same epilogues and
//    partial layout, kept as an independent cross-check of the tensor-core kernel.
// The int8-weight variant of the tensor-core kernel is in gemm8.cu.
#include "gemm_common.cuh"

namespace rk {

// The items of CTA c: its phase-0 items (two-phase launches: items [0, n0)
// spread over CTAs [0, g0)), then its phase-1 items (items [n0, nitems) spread
// over CTAs [0, p1a) and [p1b, G), numbered in that order).  A single-phase
// launch has n0 = 0.
struct ItemSpan {
    int a0, a1, b0, b1;
    __device__ __forceinline__ void init(const GemmParams &p, int c, int G) {
        const int n0 = p.n0, n1 = p.nitems - p.n0;
        a0 = a1 = 0;
        if (c < p.g0) {
            a0 = item_first(c, p.g0, n0);
            a1 = item_first(c + 1, p.g0, n0);
        }
        b0 = b1 = n0;
        const int v = c < p.p1a ? c : (c >= p.p1b ? c - p.p1b + p.p1a : -1);
        const int G1 = p.p1a + G - p.p1b;
        if (v >= 0) {
            b0 = n0 + item_first(v, G1, n1);
            b1 = n0 + item_first(v + 1, G1, n1);
        }
    }
    __device__ __forceinline__ int count() const { return (a1 - a0) + (b1 - b0); }
    __device__ __forceinline__ int at(int k) const { return k < a1 - a0 ? a0 + k : b0 + (k - (a1 - a0)); }
};

// Bounded wait until *ctr >= target (acquire), giving up after WAIT_LIMIT_NS or
// once *abort is set.
__device__ __forceinline__ bool wait_count(const uint32_t *ctr, uint32_t target, volatile uint32_t *abort) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
    if (v >= target) return true;
    const uint64_t t0 = gtimer();
    for (uint32_t it = 1;; ++it) {
        __nanosleep(100);
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
        if (v >= target) return true;
        if ((it & 15u) == 0) {
            if (*abort) return false;
            if (gtimer() - t0 > WAIT_LIMIT_NS) return false;
        }
    }
}
__device__ __forceinline__ bool check_count(const uint32_t *ctr, uint32_t target) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
    return v >= target;
}
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

__global__ void __launch_bounds__(GEMM_TC_THREADS, 1) gemm_tc_kernel(const __grid_constant__ GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    // Segment descriptors and sparsity flags are staged in shared memory and the
    // scalars in registers: the parameter block is only addressed for the tensor
    // maps, so nothing in the loops re-reads it.
    __shared__ GemmSeg sseg[GEMM_MAX_SEG];
    __shared__ uint32_t snz[MAX_NZ_BLOCKS];
    __shared__ uint64_t flags_ready;
    __shared__ uint32_t s_ok, s_last;
    uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int S = p.stages, B = p.B, npad = p.npad, NB = p.accbufs, nseg = p.nseg, n0 = p.n0, ndep = p.ndep;
    const uint32_t dep_target = (uint32_t)p.dep_target;
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
    ItemSpan span;
    span.init(p, c, G);
    const int nmine = span.count();
    if (threadIdx.x == 0) tl_start(p.tl);
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
    // still holds tensor memory on this SM: the first npre stages of this CTA in
    // walk order.  The sparsity flags of a skipping launch are known only later
    // (after the dependency wait, or in a two-phase launch after phase 0), so
    // the first npre1 stages of the phase-1 items are never skipped: their
    // activations are then zero and the products add nothing.  Every role
    // computes the same npre and npre1.
    int npre = 0, npre1 = 0;
    for (int k = 0; k < nmine; ++k) {
        const Item it = locate_item(sseg, nseg, span.at(k));
        const int ns = (it.kb1 - it.kb0) / KB_STAGE;
        npre += ns;
        if (span.at(k) >= n0) npre1 += ns;
    }
    npre = min(min(npre, S), p.prefetch);
    npre1 = min(npre1, S);
    if (warp == 0 && lane == 0) {
        for (int i = 0; i < p.nmaps; ++i) prefetch_tmap(&p.maps[i]);
        const uint64_t polW = policy_evict_first();
        int w = 0;
        for (int k = 0; k < nmine && w < npre; ++k) {
            const Item it = locate_item(sseg, nseg, span.at(k));
            const int tb = sseg[it.s].tile_base + it.tile * sseg[it.s].kb;
            const CUtensorMap *wm = &p.maps[sseg[it.s].wmap];
            for (int kb = it.kb0; kb < it.kb1 && w < npre; kb += KB_STAGE, ++w) {
                mbar_expect_tx(&full[w], W_STAGE_BYTES + XB);
                tma_load_3d(sW + (size_t)w * W_STAGE_BYTES, wm, &full[w], 0, 0, tb + kb, polW);
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
            tl_release(p.tl);
            bool ok = true;
            bool dep_ok = dep_target == 0u, flags_ok = !has_skip;
            // phase-1 stages whose weights are requested but whose activations
            // wait for phase 0 (at most S of them: the ring)
            int pend_kb[8], pend_s[8], pend_st[8], npend = 0;
            auto load_x = [&](int s_, int kb, int st) {
                const CUtensorMap *xm = &p.maps[sseg[s_].xmap];
                if (sseg[s_].x3) {
                    tma_load_3d(sX + (size_t)st * XB, xm, &full[st], 0, 0, kb, polX);
                } else {
#pragma unroll
                    for (int h = 0; h < KB_STAGE; ++h)
                        tma_load_2d(sX + (size_t)st * XB + (size_t)h * XKB, xm, &full[st], (kb + h) * GEMM_TILE_K, 0,
                                    polX);
                }
            };
            // wait for phase 0, then release the pending activation copies
            auto resolve = [&]() -> bool {
                if (!dep_ok) {
                    if (!wait_count(p.dep, dep_target, abort_flag)) return false;
                    fence_proxy_async_global();  // phase 0 wrote them through the generic proxy
                    dep_ok = true;
                }
                for (int j = 0; j < npend; ++j) load_x(pend_s[j], pend_kb[j], pend_st[j]);
                npend = 0;
                return true;
            };
            int q = 0;   // stage sequence number
            int w = 0;   // walk index (skipped stages included)
            int w1 = 0;  // walk index among phase-1 stages
            for (int k = 0; k < nmine && ok; ++k) {
                const int i = span.at(k);
                const bool ph1 = i >= n0;
                const Item it = locate_item(sseg, nseg, i);
                const int tb = sseg[it.s].tile_base + it.tile * sseg[it.s].kb;
                const CUtensorMap *wm = &p.maps[sseg[it.s].wmap];
                for (int kb = it.kb0; kb < it.kb1; kb += KB_STAGE) {
                    ++w;
                    if (ph1) {
                        const bool skippable = has_skip && w1 >= npre1;
                        ++w1;
                        if (skippable) {
                            if (!flags_ok) {  // the flags are staged once phase 0 is complete
                                if (!resolve() || !mbar_wait(&flags_ready, 0u, abort_flag)) {
                                    ok = false;
                                    break;
                                }
                                flags_ok = true;
                            }
                            if (stage_skipped(skip, kb)) continue;
                        }
                    }
                    const int st = q % S;
                    if (q >= npre) {
                        if (q >= S) {
                            if (npend == S && !resolve()) {  // the ring holds only pending stages
                                ok = false;
                                break;
                            }
                            if (!mbar_wait(&empty[st], (uint32_t)((q / S) - 1) & 1u, abort_flag)) {
                                ok = false;
                                break;
                            }
                        }
                        mbar_expect_tx(&full[st], W_STAGE_BYTES + XB);
                        tma_load_3d(sW + (size_t)st * W_STAGE_BYTES, wm, &full[st], 0, 0, tb + kb, polW);
                    }  // else: the weights were requested before the dependency wait
                    if (ph1 && !dep_ok && check_count(p.dep, dep_target)) {
                        fence_proxy_async_global();
                        dep_ok = true;
                    }
                    if (ph1 && !dep_ok) {
                        pend_kb[npend] = kb;
                        pend_s[npend] = it.s;
                        pend_st[npend] = st;
                        ++npend;
                    } else {
                        if (npend && !resolve()) {
                            ok = false;
                            break;
                        }
                        load_x(it.s, kb, st);
                    }
                    ++q;
                }
            }
            if (ok && npend && !resolve()) ok = false;
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
            bool ok = true, flags_ok = !has_skip;
            int q = 0, n = 0, w1 = 0;
            for (int k = 0; k < nmine && ok; ++k, ++n) {
                const int i = span.at(k);
                const bool ph1 = i >= n0;
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
                    if (ph1) {
                        const bool skippable = has_skip && w1 >= npre1;
                        ++w1;
                        if (skippable) {
                            if (!flags_ok) {
                                if (!mbar_wait(&flags_ready, 0u, abort_flag)) {
                                    ok = false;
                                    break;
                                }
                                flags_ok = true;
                            }
                            if (stage_skipped(skip, kb)) continue;
                        }
                    }
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
        // ------------------------------------------------ epilogue (warps 2..17)
        pdl_wait();
        const int qd = warp & 3;              // TMEM lane quarter of this warp
        const int row = qd * 32 + lane;       // accumulator row = weight row within the tile
        const int et = threadIdx.x - 64;      // 0..EPI_THREADS-1
        const int grp = et >> 7;              // column-chunk group within the lane quarter
        uint32_t *nz_out = p.nz_out;
        bool ph1_ready = false;  // phase 0 complete and the sparsity flags staged
        int n = 0, w1 = 0;
        for (int k = 0; k < nmine; ++k, ++n) {
            const int i = span.at(k);
            const bool ph1 = i >= n0;
            if (ph1 && !ph1_ready) {
                if (dep_target > 0u) {  // wait for the phase-0 items that feed phase 1 (all CTAs) to be stored
                    if (et == 0) s_ok = wait_count(p.dep, dep_target, abort_flag) ? 1u : 0u;
                    named_bar(3, EPI_THREADS);
                    const bool ok_dep = s_ok != 0u;
                    named_bar(3, EPI_THREADS);
                    if (!ok_dep) {
                        if (et == 0) {
                            *abort_flag = 1u;
                            atomicOr(p.err, ERR_TIMEOUT);
                        }
                        break;
                    }
                }
                if (has_skip) {  // stage the k-block flags of the skipping segment
                    const GemmSeg &ks = sseg[p.skip_seg];
                    const int nkb = ks.kb < MAX_NZ_BLOCKS ? ks.kb : MAX_NZ_BLOCKS;  // padded count
                    const int nreal = (ks.K + GEMM_TILE_K - 1) / GEMM_TILE_K;     // flags written
                    for (int j = et; j < nkb; j += EPI_THREADS) snz[j] = j < nreal ? __ldcg(p.nz_skip + j) : 0u;
                    named_bar(1, EPI_THREADS);
                    if (et == 0) mbar_arrive(&flags_ready);
                }
                ph1_ready = true;
            }
            const Item it = locate_item(sseg, nseg, i);
            const GemmSeg sg = sseg[it.s];  // register copy
            const int buf = n % NB;
            bool valid = !ph1;
            for (int kb = it.kb0; kb < it.kb1 && ph1; kb += KB_STAGE)
                if (w1++ < npre1 || !has_skip || !stage_skipped(skip, kb)) valid = true;
            const int nrow = it.tile * GEMM_TILE_M + row;
            const float bias = epi_bias(sg, nrow);  // in flight while the accumulator fills
            // thread 0 waits and tells the others, so that all threads take
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
            const bool nzany = epi_item(sseg[it.s], taddr, valid, nrow, it.split, npad, B, grp * EPI_CW, bias);
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
            if (i < ndep) {  // a phase-0 item that feeds phase 1 is stored: count it (release)
                named_bar(3, EPI_THREADS);
                if (sg.S > 1 && sg.fix_out != nullptr) {
                    // split: the tile's last item to arrive adds the slabs and
                    // finishes the tile, then counts it
                    if (et == 0) {
                        __threadfence();
                        const uint32_t prev = atomicAdd(sg.fix_ctr + it.tile, 1u);
                        s_last = prev == (uint32_t)(sg.S - 1) ? 1u : 0u;
                        __threadfence();
                    }
                    named_bar(3, EPI_THREADS);
                    if (s_last != 0u) {
                        fix_item(sseg[it.s], nrow, npad, B, grp * EPI_CW);
                        named_bar(3, EPI_THREADS);
                        if (et == 0) {
                            __threadfence();
                            atomicAdd(p.dep, 1u);
                        }
                    }
                } else if (et == 0) {
                    __threadfence();
                    atomicAdd(p.dep, 1u);
                }
            }
        }
    }

    __syncwarp();  // warps 0 and 1 reconverge (lane 0 ran the producer / MMA loop)
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0) tl_end(p.tl);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, ncols);
    }
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
    if (threadIdx.x == 0) tl_start(p.tl);
    pdl_wait();
    pdl_launch();
    if (threadIdx.x == 0) tl_release(p.tl);
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
    __syncthreads();
    if (threadIdx.x == 0) tl_end(p.tl);
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
