// gemm8.cu -- the int8-weight variant of the skinny projection GEMM (see the
// kernel comment below); the fp16 kernel and the shared epilogue are in gemm.cu
// and gemm_common.cuh.
#include "gemm_common.cuh"

namespace rk {

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
    if (threadIdx.x == 0) tl_start(p.tl);
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
            tl_release(p.tl);
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
            const bool nzany = epi_item(sseg[it.s], taddr, valid, nrow, it.split, npad, B, grp * EPI_CW,
                                        epi_bias(sseg[it.s], nrow));
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
    if (threadIdx.x == 0) tl_end(p.tl);
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
    {
        cudaError_t r = ensure_smem_attr((const void *)gemm_tc8_kernel, gemm_tc_max_smem());
        if (r != cudaSuccess) {
            *e = r;
            return;
        }
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

}  // namespace rk
